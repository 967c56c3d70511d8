// NVTX ranges around the library's host-side phases (a step, each bucket's
// launch, a layer gather or fetch), so that a timeline tool attached to the
// process shows which launches belong to which step and bucket.  NVTX v3 is
// header-only: without a tool attached each range costs a few nanoseconds.
#pragma once

#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

namespace zg {

class NvtxRange {
public:
    // `payload` < 0: none; else shown with the range (a bucket, layer or stage).
    explicit NvtxRange(const char* name, int64_t payload = -1)
    {
        nvtxEventAttributes_t a = {};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        if (payload >= 0) {
            a.payloadType = NVTX_PAYLOAD_TYPE_INT64;
            a.payload.llValue = payload;
        }
        nvtxRangePushEx(&a);
    }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace zg
