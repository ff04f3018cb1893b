// placement.h -- internal interface of the scale-placement checker (placement.cu).
#pragma once

#include <cuda_runtime.h>

namespace mxg {

// Validated arguments only (the C ABI checks them): k in 1..4, npairs >= 1,
// device arrays sa[npairs], sb[npairs], counts[3 * npairs], first_diff[npairs].
cudaError_t launch_placement_scan(int k, const int *sa, const int *sb, int npairs, long long *counts,
                                  long long *first_diff, int num_sms, cudaStream_t s);

}  // namespace mxg
