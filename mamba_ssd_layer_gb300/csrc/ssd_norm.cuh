// ssd_norm.cuh -- the output gate and extra normalization (ssd_norm.cu), as the C entry points see it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ssd {

// most channels (H * P) of a token the kernel handles
int64_t norm_max_channels();
// out = RMSNorm per group of (y * silu(z)) * weight over `rows` tokens of `channels` bf16 channels (z null: no
// gate; weight null: ones); two persistent CTAs per SM, enqueued on `stream`
cudaError_t launch_gated_rmsnorm(const void* y, const void* z, const float* weight, float eps, int64_t rows,
                                 int64_t channels, int groups, void* out, int num_sms, cudaStream_t stream);

}  // namespace ssd
