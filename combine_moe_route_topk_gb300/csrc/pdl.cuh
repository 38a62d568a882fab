// Programmatic dependent launch (sm_90+): every kernel of the library is
// launched with programmatic stream serialization, so the next kernel in the
// stream can be scheduled while the current one drains.  A kernel must call
// grid_dependency_wait() before it touches global memory that an earlier
// kernel in the stream reads or writes; the wait returns once every
// prerequisite grid has completed and its writes are visible.
// grid_launch_dependents() only allows the next kernel to be scheduled
// early; it never makes unfinished results visible.
#pragma once

#include <cuda_runtime.h>

namespace moe {

__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch attribute enabling programmatic stream serialization.
inline cudaLaunchAttribute pdl_attribute() {
    cudaLaunchAttribute a;
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
    return a;
}

}  // namespace moe
