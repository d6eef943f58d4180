// ol_launch.h -- host-side launch interface between the C ABI (ol_api.cpp)
// and the kernels' translation units: launchers, the tensor-core paths'
// support checks and their per-variant resource figures. Host declarations
// only; the kernels' device code does not depend on this file.
#pragma once

#include "ol_internal.h"

namespace ol {

cudaError_t launch_hpaged_quantize(const QuantizeParams& p, cudaStream_t s);
cudaError_t launch_hpaged_append(const AppendParams& p, cudaStream_t s);

// ol_decode_step; with check_only every check runs and nothing is recorded or
// launched (OL_OK: the call would enqueue its launch).
ol_status decode_step_impl(int32_t layout, const void* cache_desc, void* updated, const void* q, int32_t q_heads,
                           const void* new_kv, const int32_t* lens_host, const int32_t* lens_dev, float scale,
                           int32_t window, void* out, int32_t out_dtype, void* workspace, size_t ws_bytes,
                           ol_stream stream, bool check_only);

// Launchers (return cudaSuccess or the launch error).
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
cudaError_t launch_generic_attention(const AttnParams& p, cudaStream_t s);
// Tensor-core paths; return cudaErrorNotSupported when the shape is outside them.
bool fast_bf16_supported(const AttnParams& p);
int fast_bf16_smem(int variant);
int fast_bf16_warps(int variant);
int fast_bf16_max_cluster(int variant, bool paged);
int fast_bf16_active_clusters(int variant, bool paged, int cs);  // clusters of cs CTAs resident at once
cudaError_t launch_fast_bf16(const AttnParams& p, cudaStream_t s);
bool fast_int4_supported(const AttnParams& p);
int fast_int4_smem(int variant);
int fast_int4_warps(int variant);
int fast_int4_ctas_per_sm(int variant, bool chunk);
int fast_int4_max_cluster(int variant);
cudaError_t launch_fast_int4(const AttnParams& p, cudaStream_t s);
bool fast_hpaged_supported(const AttnParams& p);
int fast_hpaged_ctas_per_sm(bool chunk);
cudaError_t launch_fast_hpaged(const AttnParams& p, cudaStream_t s);

}  // namespace ol
