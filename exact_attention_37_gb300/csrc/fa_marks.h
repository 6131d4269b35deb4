// Stream marks between the kernels of one backward pass, for the library's own
// host-buffer pipeline: it asks for an event recorded on the launching stream as
// soon as the kernel that writes the final dK and dV has been enqueued (the dK/dV
// kernel at d = 64 and 128, the single backward launch at d = 256), so that the
// copies of dK and dV to the host can overlap the dQ kernel.
#pragma once

#include <cuda_runtime.h>

namespace fa {

// Arms (ev != nullptr) or disarms (nullptr) the mark for the calling thread.  The
// next backward pass this thread enqueues records `ev` after its dK/dV kernel.
void arm_dkdv_mark(cudaEvent_t ev);
// True once the armed event has been recorded; disarms the mark either way.
bool take_dkdv_mark();

}  // namespace fa
