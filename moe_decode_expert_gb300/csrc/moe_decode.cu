// moe_decode.cu — the whole T = 1 decode MoE block in one kernel launch.
//
// What it computes ("BI-V100 inference work log", Parts 3, 4, 9, 10):
// router GEMV + softmax + top-k, the direct-routed W13 GEMV that reads only
// the selected experts' rows in place (W13[expert_ids[k], row, :]) with
// SiluAndMul fused into it, the W2 GEMV W2[expert_ids[k], h, :] fused with
// the routing-weighted sum, and the shared expert (gate_up, SiluAndMul, down,
// optional sigmoid gate) fused into the same pass.
//
// How (GB300 design, not the pages' BI-V100 kernels): one CTA per SM, each
// owning a slice of every phase, all phases in one launch.
//   phase 1  routing-independent rows — router rows, the shared gate row and
//            the shared expert's gate/up pairs — as one CTA GEMV on m16n8k16
//            tensor-core steps (weight rows = A, x = column 0 of B), columns
//            split over the warps; the first loads go out before the PDL wait
//            when the weights are static.  Results are published as
//            (value, epoch) exchange words.
//   phase 2  every CTA gathers the E logits (one L2 round trip once they are
//            all published) and ranks them itself (fp32, lower index wins
//            ties): per-warp top-k, then an exact ranking of the candidates;
//            warp 0 forms the routing weights.  No grid barrier, no second
//            kernel.
//   phase 3  this CTA's share of the k*I routed gate/up pairs (a CTA GEMV as
//            in phase 1, or two pairs in flight per warp on wide shapes),
//            SiLU*up times the routing weight published per pair; meanwhile
//            each warp copies (cp.async) the W2 columns it needs in phase 4
//            into padded shared-memory rows.
//   phase 4  after an arrival counter shows every CTA's activations out, each
//            warp gathers the activations of its column range, splits them
//            into two storage-type terms and runs m16n8k16 steps over its
//            W2 columns: out[h] = sum_j w_j (W2_j act_j) + g (Ws2 sact) for
//            this CTA's output rows, the warps' partial rows summed in order.
// Each exchange wait is bounded by the GPU global timer and records an
// error instead of hanging.  The kernel triggers programmatic dependent launch
// at entry so the next call on the stream launches early and waits in its own
// prologue.

#include <atomic>
#include <type_traits>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kChunks = 8;  // 16-byte chunks per lane per row kept in flight

// Phase trace (built only with -DMOE_PHASE_TRACE, into a separate library):
// the ring of per-launch stamp records both T = 1 kernels write.
#ifdef MOE_PHASE_TRACE
__device__ uint64_t g_moe_trace[kTraceLaunches * kTraceCtas * kTraceSlots];
static std::atomic<unsigned> g_trace_next{0};  // ring position of the next launch
uint64_t* trace_next_record() {
  void* base = nullptr;
  if (cudaGetSymbolAddress(&base, g_moe_trace) != cudaSuccess) return nullptr;
  return static_cast<uint64_t*>(base) +
         static_cast<size_t>(g_trace_next++ % kTraceLaunches) * kTraceCtas * kTraceSlots;
}
#endif

struct DecodeArgs {
  const uint8_t* x;
  const uint8_t* wr;
  const uint8_t* w13;
  const uint8_t* w2;
  const uint8_t* sw13;
  const uint8_t* sw2;
  const uint8_t* swg;
  int32_t* topk_ids;
  float* topk_w;
  void* out;
  Control* ctrl;
  uint64_t* ll_logits;  // kLogitReplicas copies, ll_stride words apart
  uint64_t* ll_act;
  int H, E, k, I, Is, has_gate, norm_topk, out_dtype;
  int static_weights;  // MOE_FLAG_STATIC_WEIGHTS: weight reads may precede the PDL wait
  int residual;        // MOE_FLAG_RESIDUAL: out = x + block(x)
  int ll_stride;   // words between the copies of the logit words
  int act_stride;  // words between the copies of the activation words
  uint32_t rs_r, rs_s;  // shared-memory row strides (bytes) of the routed and shared W2 rows
  uint32_t off_xh, off_lg, off_act, off_terms, off_w2;
  uint64_t timeout_ns;
#ifdef MOE_PHASE_TRACE
  uint64_t* trace;  // this launch's record: [CTA][kTraceSlots]
#endif
};

// 16-byte streaming load of a weight chunk, or zeros without a load when
// `pred` is false (predicated, no branch).  Volatile, so loads issued before
// griddepcontrol.wait really are issued there.
__device__ __forceinline__ uint4 ld_stream16_pred(const void* p, bool pred) {
  uint4 r;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\tmov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\t"
      "mov.b32 %3, 0;\n\t@q ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "r"(static_cast<int>(pred)));
  return r;
}

// Up to two weight rows of H 2-byte elements, streamed to registers 16 bytes
// per lane per chunk (lane-strided, so a warp reads 512 contiguous bytes per
// instruction), then dotted with x held in shared memory as fp32.  The code
// is branch-free: chunks past the row end (and the second row of a one-row
// unit) load as zeros, and four partial sums per row shorten the FMA chain.
template <int DT>
struct RowPair {
  const uint8_t* r0;
  const uint8_t* r1;
  int two;   // 1: two rows, 0: one row
  int j;     // routed slot of the pair (phase 3)
  uint4 v0[kChunks], v1[kChunks];

  __device__ __forceinline__ void issue(int base, int nch, int lane) {
#pragma unroll
    for (int t = 0; t < kChunks; ++t) {
      const int c = base + lane + 32 * t;
      const bool in = c < nch;
      const size_t off = 16 * static_cast<size_t>(in ? c : 0);
      v0[t] = ld_stream16_pred(r0 + off, in);
      v1[t] = ld_stream16_pred(r1 + off, in && two);
    }
  }

  __device__ __forceinline__ void accumulate(const float* xs, int base, int nch, int lane, float (&a0)[4],
                                             float (&a1)[4]) const {
#pragma unroll
    for (int t = 0; t < kChunks; ++t) {
      const int c = min(base + lane + 32 * t, nch - 1);  // weights are zero past the end
      const float4 xa = reinterpret_cast<const float4*>(xs)[2 * c];
      const float4 xb = reinterpret_cast<const float4*>(xs)[2 * c + 1];
      float f[8], h[8];
      unpack8<DT>(v0[t], f);
      unpack8<DT>(v1[t], h);
      float& s0 = a0[t & 3];
      float& s1 = a1[t & 3];
      s0 = fmaf(f[0], xa.x, s0); s1 = fmaf(h[0], xa.x, s1);
      s0 = fmaf(f[1], xa.y, s0); s1 = fmaf(h[1], xa.y, s1);
      s0 = fmaf(f[2], xa.z, s0); s1 = fmaf(h[2], xa.z, s1);
      s0 = fmaf(f[3], xa.w, s0); s1 = fmaf(h[3], xa.w, s1);
      s0 = fmaf(f[4], xb.x, s0); s1 = fmaf(h[4], xb.x, s1);
      s0 = fmaf(f[5], xb.y, s0); s1 = fmaf(h[5], xb.y, s1);
      s0 = fmaf(f[6], xb.z, s0); s1 = fmaf(h[6], xb.z, s1);
      s0 = fmaf(f[7], xb.w, s0); s1 = fmaf(h[7], xb.w, s1);
    }
  }

  // Completes the dot products whose first batch was issued with issue(0).
  __device__ __forceinline__ void finish(const float* xs, int nch, int lane, float& d0, float& d1) {
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    accumulate(xs, 0, nch, lane, a0, a1);
    for (int base = 32 * kChunks; base < nch; base += 32 * kChunks) {  // rows longer than 4 KB
      issue(base, nch, lane);
      accumulate(xs, base, nch, lane, a0, a1);
    }
    d0 = warp_sum((a0[0] + a0[1]) + (a0[2] + a0[3]));
    d1 = warp_sum((a1[0] + a1[1]) + (a1[2] + a1[3]));
  }
};

// ---- W2 stage on the tensor cores (warp-level mma: the block is a GEMV over
// 16-row tiles, far below tcgen05's 128-row tiles)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// 8-byte shared load, or zeros without a load when `pred` is false.
__device__ __forceinline__ void lds64_pred(uint32_t addr, bool pred, uint32_t& x, uint32_t& y) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %3, 0;\n\tmov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\t"
      "@q ld.shared.v2.u32 {%0,%1}, [%2];\n\t}"
      : "=r"(x), "=r"(y)
      : "r"(addr), "r"(static_cast<int>(pred)));
}

// Predicated 16-byte asynchronous copy global -> shared (no branch).
__device__ __forceinline__ void cp_async16_pred(uint32_t dst, const void* src, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q cp.async.cg.shared.global [%0], [%1], 16;\n\t}" ::"r"(dst),
      "l"(src), "r"(static_cast<int>(pred))
      : "memory");
}


// 16-byte shared load, or zeros without a load when `pred` is false.
__device__ __forceinline__ uint4 lds128_pred(uint32_t addr, bool pred) {
  uint4 r;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\tmov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\t"
      "mov.b32 %3, 0;\n\t@q ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "r"(addr), "r"(static_cast<int>(pred)));
  return r;
}

// ---- CTA GEMV on m16n8k16 steps, split by columns over the 8 warps.
// Up to 16 rows per pass, all in one MMA tile: lane (g, t) streams 16-byte
// chunks of rows g and g + 8 (columns c0 + 32jj + 8t .. +7, jj < 8, of the
// warp's column slice) into registers, the A fragment of 16 rows x 16 columns
// per k-step; x, in the storage type in shared memory, is column 0 of B.
// Within a 16-byte chunk, elements 0-3 form one k-step and 4-7 the next, the
// same columns on both sides.  Column 0 of D holds the 16 rows' partial dot
// products (lanes with t = 0: rows g and g + 8).
template <int DT>
struct Gemv16 {
  uint4 w[2][8];  // [rows g / g + 8][chunk]

  __device__ __forceinline__ void issue(const uint8_t* r0, bool v0, const uint8_t* r1, bool v1, int c0, int cend,
                                        int t) {
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int c = c0 + 32 * jj + 8 * t;
      const bool in = c < cend;
      const size_t off = 2 * static_cast<size_t>(in ? c : 0);
      w[0][jj] = ld_stream16_pred(r0 + off, in && v0);
      w[1][jj] = ld_stream16_pred(r1 + off, in && v1);
    }
  }

  __device__ __forceinline__ void mma(uint32_t xh, int c0, int cend, int lane, float (&acc)[2][4]) const {
    const int t = lane & 3;
    const bool xl = lane < 4;  // B column 0 (n = lane / 4 = 0)
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int c = c0 + 32 * jj + 8 * t;
      const uint4 xv = lds128_pred(xh + 2 * static_cast<uint32_t>(c < cend ? c : 0), xl && c < cend);
      mma16816<DT>(acc[jj & 1], w[0][jj].x, w[1][jj].x, w[0][jj].y, w[1][jj].y, xv.x, xv.y);
      mma16816<DT>(acc[jj & 1], w[0][jj].z, w[1][jj].z, w[0][jj].w, w[1][jj].w, xv.z, xv.w);
    }
  }
};

// Lanes with t = 0 write the partial dot products of rows rg + g and
// rg + g + 8 into part[warp][...].
__device__ __forceinline__ void gemv_store_partials(float (*part)[64], int warp, int lane, int rg,
                                                    const float (&acc)[2][4]) {
  if ((lane & 3) == 0) {
    const int g = lane >> 2;
    part[warp][rg + g] = acc[0][0] + acc[1][0];
    part[warp][rg + g + 8] = acc[0][2] + acc[1][2];
  }
}

// v ~ t0 + t1 in the storage type: t0 = rn(v), t1 = rn(v - t0) (the
// difference is exact in fp32): about 16 significant bits in bf16, 22 in fp16
// (the unit roundoff of the pair is 2^-17 and 2^-22, far inside the block's
// tolerance).  term[s] packs term s of v.x (low half) and v.y.
template <int DT>
__device__ __forceinline__ void split2(float2 v, uint32_t (&term)[2]) {
  float x = v.x, y = v.y;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    uint32_t bx, by;
    float rx, ry;
    if constexpr (DT == MOE_BF16) {
      const __nv_bfloat16 hx = __float2bfloat16_rn(x), hy = __float2bfloat16_rn(y);
      bx = __bfloat16_as_ushort(hx); by = __bfloat16_as_ushort(hy);
      rx = __bfloat162float(hx); ry = __bfloat162float(hy);
    } else {
      const __half hx = __float2half_rn(x), hy = __float2half_rn(y);
      bx = __half_as_ushort(hx); by = __half_as_ushort(hy);
      rx = __half2float(hx); ry = __half2float(hy);
    }
    term[s] = bx | (by << 16);
    x -= rx;
    y -= ry;
  }
}

// DEPTH 1: one gate/up pair in flight per warp (<= 128 registers, two CTAs per
// SM fit); DEPTH 2: two pairs in flight (one CTA per SM), for configs with more
// routed pairs per CTA than warps.
// MODE 0 (kDecGeneral) carries every code path and picks at run time; MODE 1 /
// 2 (kDecNarrow / kDecWide) are for the standard shapes (E <= 256, k <= 8, one
// 16-row output tile per CTA, I and Is multiples of 16) and hold only their
// paths, with the activation gather's width fixed.  Each phase's code runs once
// per launch, so code that is never executed still costs time (fetching the
// instructions): the sharded layer is 3 % faster without it.
constexpr int kDecGeneral = 0, kDecNarrow = 1, kDecWide = 2;
template <int DT, int DEPTH, int MODE>
__global__ void __launch_bounds__(kDecThreads, 3 - DEPTH) decode_fused_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_ids[32];
  __shared__ float s_sel[32];
  __shared__ float s_w[32];
  __shared__ float s_gate;
  __shared__ uint32_t s_epoch;
  __shared__ uint32_t s_fail;
  __shared__ int s_next;                // next phase-3 work item of this CTA
  __shared__ unsigned long long s_cand[64];  // per-warp top-k candidates (64-bit rank keys)
  __shared__ __align__(16) unsigned long long s_wkey[256];  // every logit's 64-bit rank key
  __shared__ volatile int s_wready;     // routing weights and gate are in s_w / s_gate
  __shared__ float s_red[kDecWarps][64];

  float* xs = reinterpret_cast<float*>(smem);
  uint16_t* xh = reinterpret_cast<uint16_t*>(smem + a.off_xh);  // x in its storage type
  float* lg = reinterpret_cast<float*>(smem + a.off_lg);
  float* acts = reinterpret_cast<float*>(smem + a.off_act);
  uint16_t* terms = reinterpret_cast<uint16_t*>(smem + a.off_terms);
  uint8_t* w2s = smem + a.off_w2;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is;
  // Copies of the exchange words this instantiation writes: more copies spread
  // the polling CTAs over more L2 lines, which pays on the wide two-pairs-per-
  // warp shapes (full width: 19.20 -> 18.74 us) and costs on the narrow ones
  // (sharded: 10.08 -> 10.31 us), where the extra stores sit on the chain.
  constexpr int LREP = DEPTH == 2 ? kLogitReplicas : kLogitReplicas / 2;
  constexpr int AREP = DEPTH == 2 ? kActReplicas : kActReplicas / 2;
  const int h0 = static_cast<int>((static_cast<long long>(H) * cta) / G);
  const int hn = static_cast<int>((static_cast<long long>(H) * (cta + 1)) / G) - h0;
  const size_t rowb = static_cast<size_t>(H) * 2;
  const int nch = H >> 3;
  const int P = k * I;
  const int K = P + Is;  // columns of the concatenated [routed | shared] activation vector
  uint8_t* w2sh = w2s + static_cast<size_t>(k) * hn * a.rs_r;  // shared expert's rows
  const uint32_t w2a = smem_u32(w2s), w2sha = smem_u32(w2sh);
  const int mtiles = (hn + 15) >> 4;  // <= 4 (checked on the host)

  // Phase 4 is split by columns: warp w owns the 16-column steps [ks0, ks1)
  // of K.  It copies those columns of its W2 rows, gathers those activations
  // and runs those tensor-core steps, so only the final sum crosses warps.
  const int ksteps = (K + 15) >> 4;
  const int kpw = (ksteps + kDecWarps - 1) / kDecWarps;
  const int ks0 = min(warp * kpw, ksteps), ks1 = min(ks0 + kpw, ksteps);
  const float inv_I = 1.0f / static_cast<float>(I);
  // The expert slot (k = shared) and column within it of absolute column c.
  auto locate = [&](int c, int& j, int& i) {
    const int jr = min(k - 1, __float2int_rz((static_cast<float>(c) + 0.5f) * inv_I));
    j = c < P ? jr : k;
    i = c < P ? c - jr * I : c - P;
  };
  // Copies of this warp's W2 columns (routed: shared == false; shared expert:
  // shared == true), expert block by expert block: within a block the rows x
  // 16-byte chunks are spread over the lanes (flat index, fp32-reciprocal
  // quotient, exact for these sizes).
  const int wc0 = ks0 * 16, wc1 = min(ks1 * 16, K);  // this warp's columns
  auto copy_w2_cols = [&](bool shared) {
    int lo = shared ? max(wc0, P) : wc0;
    const int hi = shared ? wc1 : min(wc1, P);
    while (lo < hi) {
      int j, i0;
      locate(lo, j, i0);
      const int seg = min(hi, j < k ? (j + 1) * I : K) - lo;  // columns in this block
      const int nck = seg >> 3;                               // 16-byte chunks per row
      const float inv = 1.0f / static_cast<float>(nck);
      const uint32_t rs = j < k ? a.rs_r : a.rs_s;
      const uint32_t dst0 = (j < k ? w2a + static_cast<uint32_t>(j * hn) * a.rs_r : w2sha) + 2 * i0;
      const size_t srow = static_cast<size_t>(j < k ? I : Is) * 2;
      const uint8_t* src0 = (j < k ? a.w2 + (static_cast<size_t>(s_ids[min(j, k - 1)]) * H + h0) * srow
                                   : a.sw2 + static_cast<size_t>(h0) * srow) + 2 * i0;
      for (int qq = lane; qq < hn * nck; qq += 32) {
        const int r = __float2int_rz((static_cast<float>(qq) + 0.5f) * inv);
        const int c = qq - r * nck;
        cp_async16_pred(dst0 + static_cast<uint32_t>(r) * rs + 16 * c, src0 + r * srow + 16 * c, true);
      }
      lo += seg;
    }
  };

  MOE_STAMP(0);  // entry
  if (tid == 0) {
    s_fail = 0;
    s_next = 0;
    s_wready = 0;
  }
  // x and the epoch word are read right after the PDL wait; start their DRAM
  // trips now (into L2 only, so the wait still orders the reads that count).
  if (tid < ((H * 2 + 127) >> 7)) prefetch_l2(a.x + 128 * static_cast<size_t>(tid));
  if (tid == kDecThreads - 1) prefetch_l2(&a.ctrl->gen);
  pdl_launch_dependents();
  __syncthreads();

  // ---- phase 1: routing-independent rows of this CTA — its router rows
  // u = cta + qG < E (and the shared gate row), then its shared-expert pairs
  // (gate rows, then up rows) — as one CTA GEMV; the first pass's loads go out
  // before x is staged (and, with static weights, before the PDL wait).
  const int g = lane >> 2, t = lane & 3;
  const int E1 = E + a.has_gate;
  const int n1 = E1 + Is;
  const int nL = cta < E1 ? (E1 - 1 - cta) / G + 1 : 0;  // logit rows
  const int nU = cta < n1 ? (n1 - 1 - cta) / G + 1 : 0;
  const int nS = nU - nL;                                  // shared pairs
  const int R1 = nL + 2 * nS;                              // <= 64 (checked on the host)
  auto p1_row = [&](int r, bool& valid) -> const uint8_t* {
    valid = r < R1;
    const int rr = r - nL;
    const int pi = rr < nS ? rr : rr - nS;
    const int uL = min(cta + r * G, E);
    const int i = max(0, cta + (nL + pi) * G - E1);
    const uint8_t* pl = uL < E ? a.wr + static_cast<size_t>(uL) * rowb : a.swg;
    const uint8_t* ps = a.sw13 + static_cast<size_t>(rr < nS ? i : Is + i) * rowb;
    return !valid ? a.wr : (r < nL ? pl : ps);
  };
  const int cpw = ((H + 255) >> 8) * 32;  // columns per warp (H / 8, rounded up to 32)
  const int c0w = min(warp * cpw, H), cendw = min(c0w + cpw, H);
  const int cb1 = min(c0w + 256, cendw);  // end of the first 256-column batch
  const uint32_t xha = smem_u32(xh);
  Gemv16<DT> gv;
  bool va, vb;
  const uint8_t* ra = p1_row(g, va);
  const uint8_t* rb = p1_row(g + 8, vb);
  // With DEPTH 2 (one CTA per SM, so a CTA starts only when its SM frees up)
  // the shared expert's W2 copies go out in phase 3 with the routed ones,
  // keeping the work before the wait short (full-width layer 20.08 -> 19.75 us).
  if (a.static_weights) {
    gv.issue(ra, va, rb, vb, c0w, cb1, t);
    if (DEPTH == 1 && Is > 0) copy_w2_cols(true);
  }
  pdl_wait();  // x (and anything else an earlier kernel wrote) is visible from here
  MOE_STAMP(1);  // PDL wait released
  if (!a.static_weights) gv.issue(ra, va, rb, vb, c0w, cb1, t);

  uint32_t gen_prev = 0;
  if (tid == 0) gen_prev = ld_relaxed_u32(&a.ctrl->gen);  // in flight together with x
  for (int c = tid; c < nch; c += kDecThreads) {
    const uint4 raw = ld_ordered16(a.x + 16 * static_cast<size_t>(c));
    *reinterpret_cast<uint4*>(xh + 8 * c) = raw;
    float f[8];
    unpack8<DT>(raw, f);
    reinterpret_cast<float4*>(xs)[2 * c] = make_float4(f[0], f[1], f[2], f[3]);
    reinterpret_cast<float4*>(xs)[2 * c + 1] = make_float4(f[4], f[5], f[6], f[7]);
  }
  if (tid == 0) {
    uint32_t ep = gen_prev + 1u;
    s_epoch = ep ? ep : 1u;
    // The arrival counter of the other parity was last used by the previous
    // launch, which has completed; clear it for the next launch.
    if (cta == 0) atomicExch(&a.ctrl->arrive[(s_epoch + 1u) & 1u], 0u);
  }
  if (DEPTH == 1 && !a.static_weights && Is > 0) copy_w2_cols(true);
  __syncthreads();
  const uint32_t epoch = s_epoch;
  MOE_STAMP(2);  // x staged

  for (int rg = 0; rg < R1; rg += 16) {
    float acc[2][4] = {};
    for (int cb = c0w; cb < cendw; cb += 256) {
      if (rg > 0 || cb > c0w) {
        ra = p1_row(rg + g, va);
        rb = p1_row(rg + 8 + g, vb);
        gv.issue(ra, va, rb, vb, cb, min(cb + 256, cendw), t);
      }
      gv.mma(xha, cb, min(cb + 256, cendw), lane, acc);
    }
    gemv_store_partials(s_red, warp, lane, rg, acc);
  }
  __syncthreads();
  MOE_STAMP(3);  // phase-1 dot products summed
  // Every CTA reads all logits and every activation, so each word is
  // published in several copies (readers spread over more L2 lines):
  // LREP threads per result, one copy each.
  for (int o = tid / LREP; o < nL + nS; o += kDecThreads / LREP) {
    const int rep = tid % LREP;
    const bool logit = o < nL;
    const int pi = o - nL;
    const int ra0 = logit ? o : nL + pi, rb0 = logit ? o : nL + nS + pi;  // the two rows combined
    float gs = 0.0f, us = 0.0f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      gs += s_red[w][ra0];
      us += s_red[w][rb0];
    }
    const float v = logit ? gs : silu_f(gs) * us;
    uint64_t* dst = logit ? a.ll_logits + static_cast<size_t>(rep) * a.ll_stride + cta + o * G
                          : a.ll_act + static_cast<size_t>(rep & (AREP - 1)) * a.act_stride + P +
                                (cta + (nL + pi) * G - E1);
    if (rep < (logit ? LREP : AREP)) ll_store(dst, v, epoch);
  }
  MOE_STAMP(4);  // phase-1 results published

  // ---- phase 2: the logits, their top-k (fp32, lower index first on ties)
  // and the routing weights.  Every logit gets a unique 64-bit key (logit
  // key, ~index).  Lane l of warp w counts how many of logits 32w..32w+31 have
  // a larger key (16 broadcast shared loads); ranks below k are the warp's
  // candidates.  The 8 warps' candidates are then ranked exactly by all
  // threads (4 threads per candidate), and candidate rank r < k fills slot r.
  if (MODE != kDecGeneral || (E <= 256 && k <= 8)) {
    if (warp == 0) {  // one warp polls the words (all warps polling floods L2)
      const uint64_t* src = a.ll_logits + static_cast<size_t>(cta % LREP) * a.ll_stride;
      const bool ok = ll_gather<8>(src, lg, E + a.has_gate, lane, 32, epoch, global_ns() + a.timeout_ns);
      if (!__all_sync(0xffffffffu, ok) && lane == 0) s_fail = kDevTimeoutLogits;
      MOE_STAMP(5);  // logits gathered
    }
    __syncthreads();
    const int i0 = warp * 32 + lane;
    const float v0 = lg[min(i0, E - 1)];              // clamped load, no branch
    const uint32_t key = i0 < E ? order_key(v0) : 0u;  // finite logits have keys > 0
    // unique 64-bit key (logit key, ~index): its rank among the warp's 32 is
    // the number of larger keys; ranks below k are the warp's candidates
    const uint64_t mk = key ? (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~i0) : 0ull;
    s_wkey[i0] = mk;
    if (lane < 8) s_cand[warp * 8 + lane] = 0ull;
    __syncwarp();
    int rk = 0;
    const ulonglong2* wk = reinterpret_cast<const ulonglong2*>(s_wkey + warp * 32);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const ulonglong2 kk = wk[j];  // same address in every lane: broadcast
      rk += (kk.x > mk ? 1 : 0) + (kk.y > mk ? 1 : 0);
    }
    if (mk != 0ull && rk < k) s_cand[warp * 8 + rk] = mk;
    __syncthreads();
    {
      const int c = tid >> 2, q4 = tid & 3;
      const uint64_t kc = s_cand[c];
      int cnt = 0;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) cnt += s_cand[4 * jj + q4] > kc ? 1 : 0;  // 4 adjacent words per load
      cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
      cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
      if (q4 == 0 && kc != 0ull && cnt < k) {
        const int id = rank_key_index(kc);
        s_ids[cnt] = id;
        s_sel[cnt] = lg[id];
      }
    }
  } else if constexpr (MODE == kDecGeneral) {
    if (warp == 0) {
      // many experts or k > 8: one warp gathers all logits and ranks them
      const int nl = E + a.has_gate;
      const uint64_t* src = a.ll_logits + static_cast<size_t>(cta % LREP) * a.ll_stride;
      const bool ok = ll_gather<8>(src, lg, nl, lane, 32, epoch, global_ns() + a.timeout_ns);
      if (__all_sync(0xffffffffu, ok)) warp_topk<32>(lg, E, k, s_ids, s_sel);
      else if (lane == 0) s_fail = kDevTimeoutLogits;
    }
  }
  __syncthreads();
  const bool ranked = s_fail == 0;  // uniform: read after the barrier
  MOE_STAMP(6);  // ranked
  // warp 0: routing weights and the shared gate (then s_wready)
  auto weights = [&]() {
    if (ranked) {
      warp_routing_weights(lg, E, s_sel, k, a.norm_topk, s_w);
      if (lane == 0) s_gate = a.has_gate ? sigmoid_f(lg[E]) : 1.0f;
      __syncwarp();
      if (cta == 0 && lane < k) {
        a.topk_ids[lane] = s_ids[lane];
        a.topk_w[lane] = s_w[lane];
      }
    }
    if (lane == 0) {
      __threadfence_block();
      s_wready = 1;
    }
    MOE_STAMP(7);  // routing weights ready
  };
  if (DEPTH == 2 && warp == 0) weights();

  // ---- phase 3: this CTA's share of the k*I routed gate/up pairs.  Warps
  // take pairs in order from a shared counter, so warp 0 (busy ranking) only
  // picks up what is left; each activation is published already multiplied
  // by its routing weight.  With DEPTH == 2 a warp keeps two pairs' rows in
  // flight at once.  A warp copies its W2 columns of the selected experts
  // while its first pair's rows are in flight.
  auto wait_flag = [&](volatile int* f) -> bool {
    const uint64_t deadline = global_ns() + a.timeout_ns;
    while (*f == 0) {
      if (global_ns() > deadline) return false;
      __nanosleep(32);
    }
    __threadfence_block();
    return true;
  };
  auto grab = [&](int n) -> int {
    int v = 0;
    if (lane == 0) v = atomicAdd(&s_next, n);
    return __shfl_sync(0xffffffffu, v, 0);
  };
  auto start_pair = [&](RowPair<DT>& r, int p) {
    const int j = p / I, i = p - j * I;
    const size_t erow = static_cast<size_t>(s_ids[j]) * 2 * I;
    r.r0 = a.w13 + (erow + i) * rowb;
    r.r1 = a.w13 + (erow + I + i) * rowb;
    r.two = 1;
    r.j = j;
    r.issue(0, nch, lane);
  };
  auto end_pair = [&](RowPair<DT>& r, int p) -> bool {
    float g, up;
    r.finish(xs, nch, lane, g, up);
    if (!wait_flag(&s_wready)) {
      if (lane == 0) s_fail = kDevTimeoutLogits;
      return false;
    }
    if (lane < AREP) ll_store(a.ll_act + static_cast<size_t>(lane) * a.act_stride + p, silu_f(g) * up * s_w[r.j], epoch);
    return true;
  };
  if constexpr (DEPTH == 1) {
    // At most 8 pairs per CTA: all of them as one CTA GEMV (gate rows, then
    // up rows), loads issued before the W2 copies and the routing weights.
    if (ranked) {
      const int np3 = cta < P ? (P - 1 - cta) / G + 1 : 0;
      auto p3_row = [&](int r, bool& valid) -> const uint8_t* {
        valid = r < 2 * np3;
        const int pi = r < np3 ? r : r - np3;
        const int p = pi * G + cta;
        const int j = min(p / I, k - 1), i = p - j * I;
        return a.w13 + (static_cast<size_t>(s_ids[j]) * 2 * I + (r < np3 ? i : I + i)) * rowb;
      };
      ra = p3_row(g, va);
      rb = p3_row(g + 8, vb);
      gv.issue(ra, va, rb, vb, c0w, cb1, t);
      if (warp == 0) weights();
      copy_w2_cols(false);
      float acc[2][4] = {};
      for (int cb = c0w; cb < cendw; cb += 256) {
        if (cb > c0w) gv.issue(ra, va, rb, vb, cb, min(cb + 256, cendw), t);
        gv.mma(xha, cb, min(cb + 256, cendw), lane, acc);
      }
      gemv_store_partials(s_red, warp, lane, 0, acc);
      __syncthreads();
      for (int o = tid / AREP; o < np3; o += kDecThreads / AREP) {
        const int rep = tid % AREP;
        float gs = 0.0f, us = 0.0f;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) {
          gs += s_red[w][o];
          us += s_red[w][np3 + o];
        }
        const int p = o * G + cta;
        const int j = min(p / I, k - 1);
        if (rep < AREP)
          ll_store(a.ll_act + static_cast<size_t>(rep) * a.act_stride + p, silu_f(gs) * us * s_w[j], epoch);
      }
    } else if (warp == 0) {
      weights();
    }
  } else if (ranked && !s_fail) {
    bool copied = false;
    {
      RowPair<DT> rp, rq;
      for (;;) {
        const int qq = grab(2);
        const int pa = qq * G + cta, pb = (qq + 1) * G + cta;
        if (pa >= P) break;
        start_pair(rp, pa);
        if (pb < P) start_pair(rq, pb);
        if (!copied) {
          if (Is > 0) copy_w2_cols(true);
          copy_w2_cols(false);
          copied = true;
        }
        if (!end_pair(rp, pa) || pb >= P) break;
        if (!end_pair(rq, pb)) break;
      }
    }
    if (!copied) {
      if (Is > 0) copy_w2_cols(true);
      copy_w2_cols(false);
    }
  }

  // ---- phase 4 (per warp): this warp's activations and W2 columns
  // The warp reads the exchange words of its columns (all requested at once,
  // re-polling any not yet published) into its range of `acts`, writes the
  // two storage-type terms of each activation (split2; the routed ones
  // already weighted, the shared ones times the gate here; fp16 scaled by a
  // power of two that puts the range's largest magnitude in [2^14, 2^15),
  // exact and undone on the sums) in B-fragment order, then runs its
  // tensor-core steps: out[h0 + r] = sum over the K columns of W2 row r times
  // the activations, A = 16 W2 rows x 16 columns (ldmatrix from the padded
  // rows), B columns 0-1 = the activation terms, fp32 accumulation.  Lane t of
  // a B fragment needs columns 2t, 2t+1, 2t+8, 2t+9 of a step, kept at
  // 4t..4t+3 of the step's 16 slots.
  // One thread per CTA counts CTAs in and waits until 5/8 of them have
  // arrived before any warp reads the activation words: every warp polling the
  // words while most CTAs are still producing floods L2 with re-reads and
  // slows the weight streams, while waiting for all G puts a full round trip
  // after the last arrival.  From 5/8 on, the gather's first round trip
  // overlaps the last CTAs' work and the epoch tags make it re-poll the words
  // not yet published (measured: 5/8 and 1/2 equally best, 1/4 and all G
  // slower).  A CTA counts itself in as soon as its activations are out; its
  // own W2 copies land while it waits.
  MOE_STAMP(8);  // thread 0's phase-3 work done
  __syncthreads();
  if (tid == 0 && !s_fail) {
    uint32_t* cnt = &a.ctrl->arrive[epoch & 1u];
    atomicAdd(cnt, 1u);
    const uint64_t deadline = global_ns() + a.timeout_ns;
    bool arrived = true;
    while (ld_relaxed_u32(cnt) < static_cast<uint32_t>((G * 5) / 8)) {
      if (global_ns() > deadline) { arrived = false; break; }
    }
    if (!arrived) s_fail = kDevTimeoutAct;
    MOE_STAMP(9);  // 5/8 of the CTAs counted in
  }
  cp_async_wait_all();  // this thread's W2 copies
  __syncthreads();
  MOE_STAMP(10);  // W2 copies landed
  {
    const int g = lane >> 2, t = lane & 3;
    const int c0 = ks0 * 16, c1 = min(ks1 * 16, K);
    const int Kp = ksteps * 16;
    bool ok = __all_sync(0xffffffffu, s_fail == 0);  // warp-uniform
    if (ok && c1 > c0) {
      const uint64_t* rep = a.ll_act + static_cast<size_t>(cta % AREP) * a.act_stride + c0;
      const uint64_t dl = global_ns() + a.timeout_ns;
      bool got;
      if constexpr (MODE == kDecNarrow) got = ll_gather<4>(rep, acts + c0, c1 - c0, lane, 32, epoch, dl);
      else if constexpr (MODE == kDecWide) got = ll_gather<16>(rep, acts + c0, c1 - c0, lane, 32, epoch, dl);
      else got = ((c1 - c0 + 1) >> 1) <= 4 * 32 ? ll_gather<4>(rep, acts + c0, c1 - c0, lane, 32, epoch, dl)
                                                 : ll_gather<16>(rep, acts + c0, c1 - c0, lane, 32, epoch, dl);
      ok = __all_sync(0xffffffffu, got);
      if (!ok && lane == 0) s_fail = kDevTimeoutAct;
    }
    MOE_STAMP(11);  // activations gathered
    __syncwarp();
    float unsc = 1.0f;
    if (ok && ks1 > ks0) {
      const float gate = s_gate;
      const float2* acts2 = reinterpret_cast<const float2*>(acts);
      float sc = 1.0f;
      if constexpr (DT == MOE_F16) {
        float mx = 0.0f;
        for (int qp = (c0 >> 1) + lane; 2 * qp < c1; qp += 32) {
          const float2 v = acts2[qp];
          const float f = 2 * qp >= P ? gate : 1.0f;
          mx = fmaxf(mx, fmaxf(fabsf(v.x * f), fabsf(v.y * f)));
        }
        const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
        int sh = amax ? 14 - (static_cast<int>(amax >> 23) - 127) : 0;
        sh = max(-100, min(100, sh));
        sc = __int_as_float((127 + sh) << 23);
        unsc = __int_as_float((127 - sh) << 23);
      }
      for (int qp = (c0 >> 1) + lane; 2 * qp < ks1 * 16; qp += 32) {
        const int pcol = 2 * qp;
        const float2 v0 = acts2[min(qp, (K >> 1) - 1)];  // clamped load, no branch
        const float f = pcol < K ? (pcol >= P ? gate : 1.0f) * sc : 0.0f;
        uint32_t tm[2];
        split2<DT>(make_float2(v0.x * f, v0.y * f), tm);
        const int w = pcol & 15;
        const int at = (pcol & ~15) + (w < 8 ? 2 * w : 2 * w - 14);
#pragma unroll
        for (int e = 0; e < 2; ++e) *reinterpret_cast<uint32_t*>(terms + static_cast<size_t>(e) * Kp + at) = tm[e];
      }
    }
    __syncwarp();  // terms and this warp's W2 copies visible to all its lanes
    MOE_STAMP(12);  // terms written
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t ta0 = smem_u32(terms) + static_cast<uint32_t>(g * Kp + 4 * t) * 2;
    const bool bl = lane < 8;  // lanes holding B columns 0-1
    float acc[4][4], acc1[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.0f;
    acc1[0] = acc1[1] = acc1[2] = acc1[3] = 0.0f;
    if (ok && (MODE != kDecGeneral || (mtiles == 1 && (I & 15) == 0 && (Is & 15) == 0))) {
      // One 16-row tile; expert blocks are whole 16-column steps, so the
      // warp walks them as uniform segments with plain pointer increments,
      // four steps of loads in flight and two accumulator chains.
      const int row = min(lrow, hn - 1);
      const uint32_t lk = (lane >> 4) * 16;
      const uint32_t roff_r = static_cast<uint32_t>(row) * a.rs_r + lk;
      const uint32_t roff_s = static_cast<uint32_t>(row) * a.rs_s + lk;
      const int spe = I >> 4, psteps = P >> 4;
      uint32_t ta = ta0 + static_cast<uint32_t>(ks0) * 32;
      int ks = ks0;
      while (ks < ks1) {
        const int j = ks < psteps ? ks / spe : k;
        const int send = min(ks1, j < k ? (j + 1) * spe : ksteps);
        uint32_t ap = j < k ? w2a + static_cast<uint32_t>(j * hn) * a.rs_r + roff_r + (ks - j * spe) * 32
                            : w2sha + roff_s + (ks - psteps) * 32;
        for (; ks + 4 <= send; ks += 4) {
          uint32_t b[4][2], av[4][4];
#pragma unroll
          for (int v = 0; v < 4; ++v) lds64_pred(ta + 32 * v, bl, b[v][0], b[v][1]);
#pragma unroll
          for (int v = 0; v < 4; ++v) ldsm_x4(ap + 32 * v, av[v][0], av[v][1], av[v][2], av[v][3]);
          mma16816<DT>(acc[0], av[0][0], av[0][1], av[0][2], av[0][3], b[0][0], b[0][1]);
          mma16816<DT>(acc1, av[1][0], av[1][1], av[1][2], av[1][3], b[1][0], b[1][1]);
          mma16816<DT>(acc[0], av[2][0], av[2][1], av[2][2], av[2][3], b[2][0], b[2][1]);
          mma16816<DT>(acc1, av[3][0], av[3][1], av[3][2], av[3][3], b[3][0], b[3][1]);
          ap += 128;
          ta += 128;
        }
        for (; ks < send; ++ks) {
          uint32_t b0, b1, a0, a1, a2, a3;
          lds64_pred(ta, bl, b0, b1);
          ldsm_x4(ap, a0, a1, a2, a3);
          mma16816<DT>(acc[0], a0, a1, a2, a3, b0, b1);
          ap += 32;
          ta += 32;
        }
      }
    } else if (MODE == kDecGeneral && ok) {
      // General shapes: up to four 16-row tiles; each lane locates the expert
      // block and column of its 8-column chunk at every step.
      for (int ks = ks0; ks < ks1; ++ks) {
        uint32_t b0, b1;
        lds64_pred(ta0 + static_cast<uint32_t>(ks) * 32, bl, b0, b1);
        int j, i;
        locate(min(ks * 16 + (lane >> 4) * 8, K - 8), j, i);  // columns past K meet zeros in B
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          if (m < mtiles) {
            const int row = min(m * 16 + lrow, hn - 1);
            const uint32_t ap = j < k ? w2a + static_cast<uint32_t>(j * hn + row) * a.rs_r + 2 * i
                                      : w2sha + static_cast<uint32_t>(row) * a.rs_s + 2 * i;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(ap, a0, a1, a2, a3);
            mma16816<DT>(acc[m], a0, a1, a2, a3, b0, b1);
          }
        }
      }
    }
    // columns 0 and 1 (lane t = 0; the other columns are zero) of rows g and g + 8
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float top = acc[m][0] + acc[m][1], bot = acc[m][2] + acc[m][3];
      if (m == 0) {  // the fast path's second accumulator chain (zeros otherwise)
        top += acc1[0] + acc1[1];
        bot += acc1[2] + acc1[3];
      }
      top += __shfl_xor_sync(0xffffffffu, top, 1);
      bot += __shfl_xor_sync(0xffffffffu, bot, 1);
      if (t == 0) {
        s_red[warp][m * 16 + g] = top * unsc;
        s_red[warp][m * 16 + g + 8] = bot * unsc;
      }
    }
    MOE_STAMP(13);  // combine steps done
  }
  __syncthreads();
  if (!s_fail) {
    if (tid < hn) {
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) sum += s_red[w][tid];
      if (a.residual) sum += xs[h0 + tid];  // x, exact in fp32
      store_out(a.out, h0 + tid, sum, a.out_dtype);
    }
    MOE_STAMP(14);  // output written
    // Every CTA has read the epoch before publishing its activations and CTA 0
    // has now seen all of them, so the next launch may use the next epoch.
    if (cta == 0 && tid == 0) atomicExch(&a.ctrl->gen, epoch);
    return;
  }
  // ---- failure path: record the error and bump the epoch (every thread's
  // W2 copies have landed: cp_async_wait_all above)
  if (tid == 0) {
    report_error(a.ctrl, s_fail, static_cast<uint32_t>(cta));
    if (cta == 0) atomicExch(&a.ctrl->gen, epoch);
  }
}

// ------------------------------------------------------------------ host side
int decode_grid(const moe_cfg_t& c) {
  // One CTA per SM; never more CTAs than routed pairs, so that every CTA
  // publishes at least one activation (the epoch hand-over relies on it).
  const int pairs = c.top_k * c.inter;
  int g = sm_count();
  if (g > pairs) g = pairs;
  return g < 1 ? 1 : g;
}

// Shared-memory row stride (bytes) of n 2-byte elements: an odd number of
// 16-byte units, so that 8 consecutive rows start in 8 different bank groups
// (conflict-free ldmatrix).
static uint32_t w2_row_stride(int n) { return static_cast<uint32_t>(((n / 8) | 1) * 16); }

static void decode_smem_layout(const moe_cfg_t& c, int G, uint32_t& off_xh, uint32_t& off_lg, uint32_t& off_act,
                               uint32_t& off_terms, uint32_t& off_w2, size_t& total) {
  const size_t H = c.hidden, E = c.n_experts, k = c.top_k, I = c.inter, Is = c.shared_inter;
  const size_t hn_max = (H + G - 1) / G;
  const size_t Kp = (k * I + Is + 15) / 16 * 16;
  size_t off = align_up(H * 4, 128);
  off_xh = static_cast<uint32_t>(off);
  off += align_up(H * 2, 128);
  off_lg = static_cast<uint32_t>(off);
  off += align_up((E + 2) * 4, 128);
  off_act = static_cast<uint32_t>(off);
  off += align_up((Kp + 2) * 4, 128);
  off_terms = static_cast<uint32_t>(off);
  off += align_up(2 * Kp * 2, 128);
  off_w2 = static_cast<uint32_t>(off);
  off += align_up(hn_max * (k * w2_row_stride(c.inter) + (Is ? w2_row_stride(c.shared_inter) : 0)), 128);
  total = off;
}

size_t decode_smem_bytes(const moe_cfg_t& c, int G) {
  uint32_t a, b, d, e, f;
  size_t t;
  decode_smem_layout(c, G, a, b, d, e, f, t);
  return t;
}

// CTAs of `kernel` (kDecThreads threads, `smem` bytes of dynamic shared
// memory) that can be resident on one SM, from the occupancy calculator;
// cached per (device, kernel, smem) under the attribute lock.
template <typename K>
static int resident_ctas_per_sm(K kernel, size_t smem) {
  struct Entry {
    int dev;
    const void* fn;
    size_t smem;
    int n;
  };
  static Entry cache[32];
  static int used = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(attr_mutex());
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].fn == reinterpret_cast<const void*>(kernel) && cache[i].smem == smem)
      return cache[i].n;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kDecThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (used < 32) cache[used++] = Entry{dev, reinterpret_cast<const void*>(kernel), smem, n};
  return n;
}

template <int DT, int DEPTH, int MODE>
static moe_status_t launch_decode_dt(const DecodeArgs& args, int G, size_t smem, cudaStream_t st) {
  auto kernel = decode_fused_kernel<DT, DEPTH, MODE>;
  if (raise_smem_limit(kernel, smem) != cudaSuccess) return check_launch("cudaFuncSetAttribute(decode)");
  // The CTAs exchange logits and activations through memory and wait for one
  // another, so all G of them must be resident at once: refuse a launch the
  // device cannot hold instead of letting its waits run into the time limit.
  const int per_sm = resident_ctas_per_sm(kernel, smem);
  if (per_sm < 0) return set_error(MOE_ERR_CUDA, "decode: occupancy query failed");
  if (static_cast<long long>(per_sm) * sm_count() < G)
    return set_error(MOE_ERR_UNSUPPORTED,
                     "decode: %d CTAs must be co-resident but only %d per SM x %d SMs fit "
                     "(%zu B of shared memory per CTA)", G, per_sm, sm_count(), smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kernel, args) != cudaSuccess) return check_launch("decode_fused_kernel");
  stat_kernels(1);
  return MOE_OK;
}

moe_status_t launch_decode_fused(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws,
                                 const WsLayout& L, cudaStream_t st) {
  const int G = decode_grid(c);
  DecodeArgs a;
  a.x = static_cast<const uint8_t*>(p.x);
  a.wr = static_cast<const uint8_t*>(p.router_w);
  a.w13 = static_cast<const uint8_t*>(p.w13);
  a.w2 = static_cast<const uint8_t*>(p.w2);
  a.sw13 = static_cast<const uint8_t*>(p.shared_w13);
  a.sw2 = static_cast<const uint8_t*>(p.shared_w2);
  a.swg = static_cast<const uint8_t*>(p.shared_gate_w);
  a.topk_ids = p.topk_ids;
  a.topk_w = p.topk_w;
  a.out = p.out;
  a.ctrl = reinterpret_cast<Control*>(ws + L.ctrl);
  a.ll_logits = reinterpret_cast<uint64_t*>(ws + L.ll_logits);
  a.ll_act = reinterpret_cast<uint64_t*>(ws + L.ll_act);
  a.H = c.hidden; a.E = c.n_experts; a.k = c.top_k; a.I = c.inter; a.Is = c.shared_inter;
  a.has_gate = c.has_shared_gate; a.norm_topk = c.norm_topk; a.out_dtype = c.out_dtype;
  a.static_weights = (c.flags & MOE_FLAG_STATIC_WEIGHTS) ? 1 : 0;
  a.residual = (c.flags & MOE_FLAG_RESIDUAL) ? 1 : 0;
  a.ll_stride = (c.n_experts + 2) & ~1;
  a.act_stride = (c.top_k * c.inter + c.shared_inter + 1) & ~1;
  a.rs_r = w2_row_stride(c.inter);
  a.rs_s = w2_row_stride(c.shared_inter);
  size_t smem;
  decode_smem_layout(c, G, a.off_xh, a.off_lg, a.off_act, a.off_terms, a.off_w2, smem);
  a.timeout_ns = wait_timeout_ns();
#ifdef MOE_PHASE_TRACE
  a.trace = trace_next_record();
  if (!a.trace) return check_launch("trace buffer");
  if (G > kTraceCtas) return set_error(MOE_ERR_UNSUPPORTED, "trace build: more than %d CTAs", kTraceCtas);
#endif
  if (smem > 227 * 1024)
    return set_error(MOE_ERR_UNSUPPORTED, "decode: needs %zu B of shared memory per CTA (max 232448)", smem);
  if (2 * ((c.n_experts + c.has_shared_gate + c.shared_inter + G - 1) / G) > 64)
    return set_error(MOE_ERR_UNSUPPORTED, "decode: more than 64 routing-independent rows per CTA");
  if ((c.hidden + G - 1) / G > 64)
    return set_error(MOE_ERR_UNSUPPORTED, "decode: %d output rows per CTA (hidden / CTAs) exceed 64",
                     (c.hidden + G - 1) / G);
  // two pairs in flight per warp when a CTA has more routed pairs than warps
  const bool deep = (c.top_k * c.inter + G - 1) / G > kDecWarps;
  // standard shapes take an instantiation without the general code paths
  const int H = c.hidden, K = c.top_k * c.inter + c.shared_inter;
  const bool standard = c.n_experts <= 256 && c.top_k <= 8 && H >= G && (H + G - 1) / G <= 16 &&
                        c.inter % 16 == 0 && c.shared_inter % 16 == 0;
  const int kpw = ((K + 15) / 16 + kDecWarps - 1) / kDecWarps;  // 16-column steps per warp
  const int mode = !standard ? kDecGeneral : ((kpw * 16 + 1) / 2 <= 4 * 32 ? kDecNarrow : kDecWide);
  if (mode == kDecGeneral) stat_decode_general();
  auto go = [&](auto dt, auto depth) -> moe_status_t {
    constexpr int D = decltype(dt)::value, P = decltype(depth)::value;
    if (mode == kDecNarrow) return launch_decode_dt<D, P, kDecNarrow>(a, G, smem, st);
    if (mode == kDecWide) return launch_decode_dt<D, P, kDecWide>(a, G, smem, st);
    return launch_decode_dt<D, P, kDecGeneral>(a, G, smem, st);
  };
  using bf = std::integral_constant<int, MOE_BF16>;
  using f16 = std::integral_constant<int, MOE_F16>;
  using d1 = std::integral_constant<int, 1>;
  using d2 = std::integral_constant<int, 2>;
  if (c.dtype == MOE_BF16) return deep ? go(bf{}, d2{}) : go(bf{}, d1{});
  return deep ? go(f16{}, d2{}) : go(f16{}, d1{});
}

}  // namespace moe

#ifdef MOE_PHASE_TRACE
// Host side of the phase trace, exported only by the trace build: geometry,
// reset (next launch records into ring entry 0; records zeroed) and read-back.
extern "C" __attribute__((visibility("default"))) int moe_trace_reset(void) {
  moe::g_trace_next = 0;
  void* base = nullptr;
  if (cudaGetSymbolAddress(&base, moe::g_moe_trace) != cudaSuccess) return 1;
  return cudaMemset(base, 0, sizeof(moe::g_moe_trace)) == cudaSuccess ? 0 : 1;
}
extern "C" __attribute__((visibility("default"))) int moe_trace_geometry(int* slots, int* ctas, int* launches) {
  *slots = moe::kTraceSlots;
  *ctas = moe::kTraceCtas;
  *launches = moe::kTraceLaunches;
  return 0;
}
extern "C" __attribute__((visibility("default"))) int moe_trace_read(uint64_t* dst, size_t words) {
  if (words > sizeof(moe::g_moe_trace) / 8) return 1;
  return cudaMemcpyFromSymbol(dst, moe::g_moe_trace, words * 8) == cudaSuccess ? 0 : 1;
}
#endif
