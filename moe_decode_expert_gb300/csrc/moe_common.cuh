// moe_common.cuh — device helpers shared by the MoE kernels (sm_103a).
//
// Streaming weight loads, fp16/bf16 unpacking, warp reductions, the warp
// top-k selector, bounded waits on the GPU global timer, the low-latency
// (value, epoch) words CTAs exchange through global memory, mbarrier and
// bulk-copy (TMA, untiled) wrappers, and programmatic-dependent-launch
// controls.  Inline PTX only; no library kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ------------------------------------------------------------------ status
// Device status codes recorded in the workspace control block (first wins).
enum : uint32_t {
  kDevOk = 0,
  kDevTimeoutLogits = 1,  // router logits of another CTA never arrived
  kDevTimeoutAct = 2,     // activations of another CTA never arrived
  kDevTimeoutCopy = 3,    // a bulk copy never completed
  kDevBadExpert = 4,      // an expert id outside [0, E)
  kDevTimeoutTest = 5,    // the test hook's wait ran out (expected)
};

// Control block at offset 0 of every workspace (256 bytes).
struct Control {
  uint32_t status;     // first device-side error code, 0 = none
  uint32_t detail;     // CTA (or token) that recorded it
  uint32_t gen;        // epoch of the last single-launch decode on this workspace
  uint32_t never_set;  // a flag no kernel writes (failure-path test)
  uint32_t arrive[2];  // CTAs done publishing activations, by launch-epoch parity
  uint32_t pad[58];
};
static_assert(sizeof(Control) == 256, "control block is 256 bytes");

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Phase trace (built only with -DMOE_PHASE_TRACE, into a separate library):
// thread 0 of each CTA stores the GPU global time at fixed points of a T = 1
// kernel into its launch's record (kernel argument `a.trace`, [CTA][slot]),
// read back by moe_trace_read.  Compiled out otherwise.
#ifdef MOE_PHASE_TRACE
constexpr int kTraceSlots = 32, kTraceCtas = 256, kTraceLaunches = 64;
#define MOE_STAMP(s)                                                          \
  do {                                                                        \
    if (threadIdx.x == 0 && blockIdx.x < kTraceCtas)                          \
      a.trace[blockIdx.x * kTraceSlots + (s)] = global_ns();                  \
  } while (0)
#else
#define MOE_STAMP(s) \
  do {               \
  } while (0)
#endif

__device__ __forceinline__ void report_error(Control* c, uint32_t code, uint32_t detail) {
  if (atomicCAS(&c->status, 0u, code) == 0u) atomicExch(&c->detail, detail);
}

// ------------------------------------------------ programmatic dependent launch
// Let the next kernel on the stream start launching (its CTAs then block in
// their own pdl_wait until this grid has completed and flushed).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the preceding kernel on the stream has completed and its memory
// operations are visible.  A no-op when launched without the PDL attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// --------------------------------------------------------------- loads
// Loads in kernels launched with programmatic dependent launch are volatile
// asm (or plain loads through pointers without __restrict__): the compiler
// then keeps them after griddepcontrol.wait.  A non-volatile asm load, or a
// load through a const __restrict__ kernel parameter (an invariant load to
// the compiler), may be scheduled above the wait and read stale data.
//
// 16-byte streaming load of read-only weights: not kept in L1, with a 256-byte
// L2 prefetch hint (consecutive lanes read consecutive 16-byte chunks).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16-byte load that the compiler keeps after every earlier volatile asm (in
// particular after griddepcontrol.wait), for data an earlier kernel may write.
__device__ __forceinline__ uint4 ld_ordered16(const void* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}

// L2-only prefetch of the 128-byte line holding p.  It never brings data into
// L1, so it may precede griddepcontrol.wait even for data the preceding kernel
// is still writing: L2 is the point of coherence and later reads see the write.
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// 16-byte asynchronous copy global -> shared through L2 only (cp.async.cg);
// completion is awaited per thread with cp_async_wait_all().  Both addresses
// 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Two 2-byte floats packed in a 32-bit word -> two fp32 (exact).
template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (DT == MOE_BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  }
}

template <int DT>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  float2 a = unpack2<DT>(v.x), b = unpack2<DT>(v.y), c = unpack2<DT>(v.z), d = unpack2<DT>(v.w);
  f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
}

template <int DT>
__device__ __forceinline__ float load_scalar(const void* base, size_t idx) {
  const uint16_t b = reinterpret_cast<const uint16_t*>(base)[idx];
  if constexpr (DT == MOE_BF16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
  else return __half2float(__ushort_as_half(b));
}

// Store one fp32 result in the output element type (round to nearest even).
__device__ __forceinline__ void store_out(void* out, size_t idx, float v, int out_dtype) {
  if (out_dtype == MOE_F32) {
    reinterpret_cast<float*>(out)[idx] = v;
  } else if (out_dtype == MOE_BF16) {
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  } else {
    reinterpret_cast<__half*>(out)[idx] = __float2half_rn(v);
  }
}

// ---------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// g * sigmoid(g) and sigmoid(s) with a correctly rounded reciprocal (no
// division slow path); expf keeps full fp32 accuracy.
__device__ __forceinline__ float silu_f(float g) { return g * __frcp_rn(1.0f + expf(-g)); }
__device__ __forceinline__ float sigmoid_f(float s) { return __frcp_rn(1.0f + expf(-s)); }

// Order-preserving map of a finite fp32 onto uint32 (larger float -> larger
// key).  Every finite value (and -inf) maps above 0, so 0 can mark "taken".
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Top-k of n <= 32*MAXM fp32 values held in shared memory, by (value desc,
// index asc).  Called by all 32 lanes of one warp.  Lane l owns the
// contiguous index range [l*m, l*m + m), so among lanes whose best keys tie,
// the lowest lane holds the lowest index; within a lane a strict '>' scan
// keeps the lowest index.  Writes out_ids[0..k) and out_vals[0..k).
template <int MAXM>
__device__ __forceinline__ void warp_topk(const float* vals, int n, int k, int* out_ids,
                                          float* out_vals) {
  const int lane = threadIdx.x & 31;
  const int m = (n + 31) >> 5;
  uint32_t key[MAXM];
#pragma unroll
  for (int s = 0; s < MAXM; ++s) {
    const int idx = lane * m + s;
    key[s] = (s < m && idx < n) ? order_key(vals[idx]) : 0u;
  }
  uint32_t bk = 0u;
  int bs = -1;
#pragma unroll
  for (int s = 0; s < MAXM; ++s)
    if (key[s] > bk) { bk = key[s]; bs = s; }
  for (int r = 0; r < k; ++r) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t ball = __ballot_sync(0xffffffffu, bs >= 0 && bk == mx);
    const int winner = __ffs(ball) - 1;
    if (lane == winner) {
      const int idx = lane * m + bs;
      out_ids[r] = idx;
      out_vals[r] = vals[idx];
#pragma unroll
      for (int s = 0; s < MAXM; ++s)
        if (s == bs) key[s] = 0u;
      bk = 0u;
      bs = -1;
#pragma unroll
      for (int s = 0; s < MAXM; ++s)
        if (key[s] > bk) { bk = key[s]; bs = s; }
    }
    __syncwarp();
  }
}

// Compare-exchange of (key, index) pairs: afterwards (ka, ia) ranks first by
// (key desc, index asc).
__device__ __forceinline__ void ce_desc(uint32_t& ka, int& ia, uint32_t& kb, int& ib) {
  const bool swap = kb > ka || (kb == ka && ib < ia);
  const uint32_t tk = swap ? kb : ka;
  const int ti = swap ? ib : ia;
  kb = swap ? ka : kb;
  ib = swap ? ia : ib;
  ka = tk;
  ia = ti;
}

// Top-k for n <= 256 values (same contract as warp_topk): each lane sorts its
// 8 (key, index) pairs once with a 19-comparator network, then every round
// takes the best lane head (redux max; lowest lane among equal heads, which
// holds the lowest index) and that lane shifts its sorted list by one.
struct NoSelectHook {
  __device__ __forceinline__ void operator()(int) const {}
};

// `on_select(r)` is called by all lanes once out_ids[r] is written (after a
// warp sync), so a caller can act on each expert while the ranking goes on.
template <class Hook = NoSelectHook>
__device__ __forceinline__ void warp_topk_sorted8(const float* vals, int n, int k, int* out_ids,
                                                  float* out_vals, Hook on_select = Hook()) {
  const int lane = threadIdx.x & 31;
  const int m = (n + 31) >> 5;  // <= 8
  uint32_t kk[8];
  int ii[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int idx = lane * m + s;
    const bool in = s < m && idx < n;
    kk[s] = in ? order_key(vals[idx]) : 0u;
    ii[s] = in ? idx : 0x7fffffff;
  }
  // optimal 8-input sorting network (19 comparators), descending
  ce_desc(kk[0], ii[0], kk[2], ii[2]); ce_desc(kk[1], ii[1], kk[3], ii[3]);
  ce_desc(kk[4], ii[4], kk[6], ii[6]); ce_desc(kk[5], ii[5], kk[7], ii[7]);
  ce_desc(kk[0], ii[0], kk[4], ii[4]); ce_desc(kk[1], ii[1], kk[5], ii[5]);
  ce_desc(kk[2], ii[2], kk[6], ii[6]); ce_desc(kk[3], ii[3], kk[7], ii[7]);
  ce_desc(kk[0], ii[0], kk[1], ii[1]); ce_desc(kk[2], ii[2], kk[3], ii[3]);
  ce_desc(kk[4], ii[4], kk[5], ii[5]); ce_desc(kk[6], ii[6], kk[7], ii[7]);
  ce_desc(kk[2], ii[2], kk[4], ii[4]); ce_desc(kk[3], ii[3], kk[5], ii[5]);
  ce_desc(kk[1], ii[1], kk[4], ii[4]); ce_desc(kk[3], ii[3], kk[6], ii[6]);
  ce_desc(kk[1], ii[1], kk[2], ii[2]); ce_desc(kk[3], ii[3], kk[4], ii[4]);
  ce_desc(kk[5], ii[5], kk[6], ii[6]);
  for (int r = 0; r < k; ++r) {
    const uint32_t mx = __reduce_max_sync(0xffffffffu, kk[0]);
    const uint32_t ball = __ballot_sync(0xffffffffu, kk[0] == mx && ii[0] != 0x7fffffff);
    const int winner = __ffs(ball) - 1;
    if (lane == winner) {
      out_ids[r] = ii[0];
      out_vals[r] = vals[ii[0]];
#pragma unroll
      for (int s = 0; s < 7; ++s) { kk[s] = kk[s + 1]; ii[s] = ii[s + 1]; }
      kk[7] = 0u;
      ii[7] = 0x7fffffff;
    }
    __syncwarp();
    on_select(r);
  }
  __syncwarp();
}

// ---- top-8 of up to 256 values by merging sorted lists across the warp.
// Each value becomes a 64-bit key, (order_key(value) << 32) | ~index, so that a
// larger key ranks first and equal values rank the lower index first; keys
// are unique.  Padding keys are 0, below every real key.
__device__ __forceinline__ uint64_t rank_key(float v, int idx) {
  return (static_cast<uint64_t>(order_key(v)) << 32) | static_cast<uint32_t>(~idx);
}
__device__ __forceinline__ int rank_key_index(uint64_t key) { return static_cast<int>(~static_cast<uint32_t>(key)); }
__device__ __forceinline__ void ce64(uint64_t& a, uint64_t& b) {  // a <- max, b <- min
  const bool sw = b > a;
  const uint64_t t = sw ? b : a;
  b = sw ? a : b;
  a = t;
}
// Sorts c[0..8) descending (bitonic merge network for a bitonic sequence).
__device__ __forceinline__ void bitonic8_desc(uint64_t (&c)[8]) {
  ce64(c[0], c[4]); ce64(c[1], c[5]); ce64(c[2], c[6]); ce64(c[3], c[7]);
  ce64(c[0], c[2]); ce64(c[1], c[3]); ce64(c[4], c[6]); ce64(c[5], c[7]);
  ce64(c[0], c[1]); ce64(c[2], c[3]); ce64(c[4], c[5]); ce64(c[6], c[7]);
}
// All 32 lanes end with c[0..8) = the 8 largest keys of vals[0..n), n <= 256,
// sorted descending.  Lane l starts from indices l, l+32, ...; its 8 keys are
// sorted (19-comparator network), then five rounds merge lane groups of 2, 4,
// ..., 32: a lane keeps the top 8 of its list and its partner's (elementwise
// max against the partner's list reversed gives a bitonic sequence holding
// them, which one bitonic merge sorts).
__device__ __forceinline__ void warp_top8_keys(const float* vals, int n, uint64_t (&c)[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int idx = s * 32 + lane;
    const uint64_t key = rank_key(vals[idx < n ? idx : n - 1], idx);  // clamped load, no branch
    c[s] = idx < n ? key : 0ull;
  }
  ce64(c[0], c[2]); ce64(c[1], c[3]); ce64(c[4], c[6]); ce64(c[5], c[7]);
  ce64(c[0], c[4]); ce64(c[1], c[5]); ce64(c[2], c[6]); ce64(c[3], c[7]);
  ce64(c[0], c[1]); ce64(c[2], c[3]); ce64(c[4], c[5]); ce64(c[6], c[7]);
  ce64(c[2], c[4]); ce64(c[3], c[5]);
  ce64(c[1], c[4]); ce64(c[3], c[6]);
  ce64(c[1], c[2]); ce64(c[3], c[4]); ce64(c[5], c[6]);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    uint64_t p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = __shfl_xor_sync(0xffffffffu, c[7 - i], m);
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = c[i] > p[i] ? c[i] : p[i];
    bitonic8_desc(c);
  }
}

// Routing weights for the k selected logits (sel[0] is the largest).  With
// norm_topk: softmax over the k selected logits, which equals the full
// softmax renormalised over the k.  Without: exp(l - max) / sum over all n.
// Called by one full warp; lane j < k writes w[j].
__device__ __forceinline__ void warp_routing_weights(const float* all, int n, const float* sel,
                                                     int k, int norm_topk, float* w) {
  const int lane = threadIdx.x & 31;
  const float mx = sel[0];
  const float ej = lane < k ? expf(sel[lane] - mx) : 0.0f;
  float z;
  if (norm_topk) {
    z = warp_sum(ej);
  } else {
    float part = 0.0f;
    for (int e = lane; e < n; e += 32) part += expf(all[e] - mx);
    z = warp_sum(part);
  }
  if (lane < k) w[lane] = ej / z;
}

// ----------------------------------------------- low-latency exchange words
// A 64-bit word carrying an fp32 value (low half) and the launch epoch (high
// half), written with one single-copy-atomic store.  A reader that sees the
// current epoch in the high half also sees the value written with it, so one
// load is both the flag check and the data read.
__device__ __forceinline__ void ll_store(uint64_t* p, float v, uint32_t epoch) {
  const uint64_t w = (static_cast<uint64_t>(epoch) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// Two consecutive exchange words (16-byte aligned) in one vector load; each
// 64-bit element is read single-copy atomically.  No "memory" clobber, so the
// compiler may issue a batch of these before using any result.
__device__ __forceinline__ ulonglong2 ll_load2(const uint64_t* p) {
  ulonglong2 w;
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0,%1}, [%2];" : "=l"(w.x), "=l"(w.y) : "l"(p));
  return w;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One exchange word at p, or zero without a load when `pred` is false.
__device__ __forceinline__ uint64_t ll_load1_pred(const uint64_t* p, bool pred) {
  uint64_t w;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\tmov.b64 %0, 0;\n\t"
      "@q ld.relaxed.gpu.global.b64 %0, [%1];\n\t}"
      : "=l"(w)
      : "l"(p), "r"(static_cast<int>(pred)));
  return w;
}

// Two exchange words at p, or zeros without a load when `pred` is false.
__device__ __forceinline__ ulonglong2 ll_load2_pred(const uint64_t* p, bool pred) {
  ulonglong2 w;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %3, 0;\n\tmov.b64 %0, 0;\n\tmov.b64 %1, 0;\n\t"
      "@q ld.relaxed.gpu.global.v2.b64 {%0,%1}, [%2];\n\t}"
      : "=l"(w.x), "=l"(w.y)
      : "l"(p), "r"(static_cast<int>(pred)));
  return w;
}

// Gather n exchange words of this epoch into dst (fp32).  `nthr` threads
// cooperate, this one being `tid`; word pairs are read with 16-byte loads
// (the word array is padded to an even length).  A thread requests all its
// pairs (up to UM per round, predicated, no branches) back to back, so the
// common case costs one L2 round trip; words not yet published are re-polled
// until `deadline` (the retry loop is warp-uniform).  Returns false if words
// were still missing then.
template <int UM>
__device__ __forceinline__ bool ll_gather(const uint64_t* src, float* dst, int n, int tid, int nthr,
                                          uint32_t epoch, uint64_t deadline) {
  const int npairs = (n + 1) >> 1;
  const int U = (npairs + nthr - 1) / nthr;
  for (int b0 = 0; b0 < U; b0 += UM) {
    ulonglong2 w[UM];
    uint32_t want = 0;
#pragma unroll
    for (int u = 0; u < UM; ++u) {
      const int q = tid + nthr * (b0 + u);
      const bool in = q < npairs;
      want |= (in ? 1u : 0u) << u;
      w[u] = ll_load2_pred(src + 2 * (in ? q : 0), in);
    }
    for (;;) {
      uint32_t missing = 0;
#pragma unroll
      for (int u = 0; u < UM; ++u) {
        const int q = tid + nthr * (b0 + u);
        const bool ok0 = static_cast<uint32_t>(w[u].x >> 32) == epoch;
        const bool ok1 = 2 * q + 1 >= n || static_cast<uint32_t>(w[u].y >> 32) == epoch;
        const bool wanted = (want >> u) & 1u;
        const bool good = wanted && ok0 && ok1;
        if (good) dst[2 * q] = __uint_as_float(static_cast<uint32_t>(w[u].x));
        if (good && 2 * q + 1 < n) dst[2 * q + 1] = __uint_as_float(static_cast<uint32_t>(w[u].y));
        missing |= (wanted && !good ? 1u : 0u) << u;
      }
      want = missing;
      if (!__any_sync(0xffffffffu, want != 0u)) break;
      if (__any_sync(0xffffffffu, global_ns() > deadline)) return false;
#pragma unroll
      for (int u = 0; u < UM; ++u) {
        const bool re = (want >> u) & 1u;
        w[u] = ll_load2_pred(src + 2 * (re ? tid + nthr * (b0 + u) : 0), re);
      }
    }
  }
  return true;
}

// ---------------------------------------------- warp-level tensor-core step
// D (16x8 fp32) += A (16x16, row-major fragment a0..a3) * B (16x8, b0..b1),
// both operands in the storage type DT.
template <int DT>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (DT == MOE_BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// ------------------------------------------------- mbarrier + bulk copies
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of `bar` to complete, or until `deadline`.
__device__ __forceinline__ bool mbar_wait_until(uint64_t* bar, uint32_t parity, uint64_t deadline) {
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() > deadline) return false;
  }
  return true;
}
// Untiled bulk copy global -> this CTA's shared memory, completing `bytes` of
// transaction count on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace moe
