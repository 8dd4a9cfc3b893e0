// mmq_pdl.cuh -- programmatic dependent launch from inside a kernel.
#pragma once

namespace mmq {

// Let the next kernel in the stream start its launch now (its CTAs still
// wait for this grid to complete before reading what it writes), and wait
// for the previous kernel in the stream to complete with its writes
// visible.  Both are no-ops for a launch without the programmatic-
// serialisation attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

}  // namespace mmq
