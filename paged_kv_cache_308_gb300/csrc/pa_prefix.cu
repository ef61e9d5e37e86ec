// Chunked-prefill ("prefix") attention kernels over the paged cache: the
// warp-level MMA kernel (pa_prefix_kernel.cuh) and the tcgen05 / tensor-memory
// kernel (pa_prefix_tc.cuh), with their launchers.
#include "pa_prefix.h"

#include <math.h>

#include "pa_decode.h"
#include "pa_device.cuh"

namespace pa {

#include "pa_prefix_kernel.cuh"
#include "pa_prefix_tc.cuh"

}  // namespace pa
