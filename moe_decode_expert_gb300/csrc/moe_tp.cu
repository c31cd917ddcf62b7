// moe_tp.cu — the sum of per-shard partial outputs for tensor-parallel MoE.
//
// Tensor parallelism as the pages run their model ("BI-V100 inference work
// log", Part 2: TP = 4 splits the expert intermediate size I = 512 into 128
// per GPU; Part 9 and the decode report's module profiling: one all-reduce of
// the MoE output per layer): every shard holds a slice of the intermediate
// dimension of every expert (and of the shared expert), routes the token
// itself with the replicated router, and produces a partial output that is
// exact to sum.  With out_dtype = MOE_F32 the decode and grouped calls emit
// those partials in fp32; this kernel adds them (in shard order, so the
// result does not depend on timing), optionally adds the residual x, and
// rounds once to the output type.  Across GPUs the partials are first summed
// by an all-reduce, then this call (n_parts = 1) finishes them.

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

// out[i] = (sum over p of parts[p * n + i]) (+ x[i]), four elements per thread.
__global__ void __launch_bounds__(256) sum_partials_kernel(const float* parts, int n_parts, int64_t n4, int64_t n,
                                                           const uint16_t* xres, int x_dtype, void* out,
                                                           int out_dtype) {
  pdl_launch_dependents();
  pdl_wait();  // the partials come from the preceding kernels on the stream
  const int64_t q = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (q >= n4) return;
  const float4* p4 = reinterpret_cast<const float4*>(parts);
  float4 acc = p4[q];
  for (int p = 1; p < n_parts; ++p) {
    const float4 v = p4[static_cast<int64_t>(p) * (n >> 2) + q];
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  const int64_t o = 4 * q;
  if (xres) {
    const uint2 r = *reinterpret_cast<const uint2*>(xres + o);
    const float2 a = x_dtype == MOE_BF16 ? unpack2<MOE_BF16>(r.x) : unpack2<MOE_F16>(r.x);
    const float2 b = x_dtype == MOE_BF16 ? unpack2<MOE_BF16>(r.y) : unpack2<MOE_F16>(r.y);
    acc.x += a.x; acc.y += a.y; acc.z += b.x; acc.w += b.y;
  }
  store_out(out, o, acc.x, out_dtype);
  store_out(out, o + 1, acc.y, out_dtype);
  store_out(out, o + 2, acc.z, out_dtype);
  store_out(out, o + 3, acc.w, out_dtype);
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_sum_partials(const float* partials, int32_t n_parts, int64_t n, const void* residual,
                                         int32_t residual_dtype, void* out, int32_t out_dtype, void* stream) {
  if (!partials || !out) return set_error(MOE_ERR_INVALID_ARG, "partials / out is NULL");
  if (n_parts < 1) return set_error(MOE_ERR_INVALID_ARG, "n_parts must be >= 1");
  if (n < 0 || n % 8) return set_error(MOE_ERR_INVALID_ARG, "n must be a non-negative multiple of 8");
  if ((reinterpret_cast<uintptr_t>(partials) | reinterpret_cast<uintptr_t>(out) |
       reinterpret_cast<uintptr_t>(residual)) & 15u)
    return set_error(MOE_ERR_INVALID_ARG, "partials, out and residual must be 16-byte aligned");
  if (out_dtype != MOE_F16 && out_dtype != MOE_BF16 && out_dtype != MOE_F32)
    return set_error(MOE_ERR_UNSUPPORTED, "out_dtype must be MOE_F16, MOE_BF16 or MOE_F32");
  if (residual && residual_dtype != MOE_F16 && residual_dtype != MOE_BF16)
    return set_error(MOE_ERR_UNSUPPORTED, "residual_dtype must be MOE_F16 or MOE_BF16");
  if (n == 0) return MOE_OK;
  const int64_t n4 = n / 4;
  const int64_t blocks = (n4 + 255) / 256;
  if (blocks > 0x7fffffff) return set_error(MOE_ERR_UNSUPPORTED, "n too large");
  if (launch_pdl(sum_partials_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                 static_cast<cudaStream_t>(stream), partials, n_parts, n4, n,
                 static_cast<const uint16_t*>(residual), residual_dtype, out, out_dtype) != cudaSuccess)
    return check_launch("sum_partials_kernel");
  stat_kernels(1);
  return MOE_OK;
}
