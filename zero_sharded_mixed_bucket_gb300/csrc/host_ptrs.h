// Host-side query: are all of these pointers device memory of the current
// GPU?  The kernels that copy tiles out with bulk asynchronous copies use
// them only for destinations in device memory, and the layer gather's
// chunked order (which reads each chunk's source once per destination) only
// for sources and destinations there; pinned or other host memory (which
// the library also accepts) keeps the per-thread store kernels.
#pragma once

#include <cuda_runtime.h>

namespace zg {

// Pointer kinds are asked of the driver on every call (an address the
// caller freed may later be host or managed memory) and remembered per
// thread for stream capture: while `stream` is being captured into a graph
// no query is made (it could invalidate the capture), remembered answers
// are used and an unknown pointer counts as not device memory.
bool device_resident(void* const* ptrs, int n, cudaStream_t stream);

}  // namespace zg
