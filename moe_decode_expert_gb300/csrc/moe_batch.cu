// moe_batch.cu — the decode MoE block for 2 <= T <= 16 tokens in one launch.
//
// What it computes: the block of the T = 1 kernel for each of T tokens
// ("BI-V100 inference work log", Parts 3, 4, 9, 10): router GEMV, softmax and
// top-k per token, the direct-routed gate/up GEMV with SiluAndMul, the down
// GEMV with the routing-weighted sum and the shared expert; with the tokens
// grouped per expert so that each selected expert's weights stream from HBM
// once per step (Part 7; "Decode throughput analysis report", the tiny-batch
// MoE fast path).
//
// How (GB300 design): one CTA per SM, every phase in one launch, the CTAs
// exchanging (value, epoch) words through global memory with bounded waits
// (no grid barrier, no second kernel).  The weight GEMVs run on m16n8k16
// tensor-core steps whose B columns are the tokens: one weight stream serves
// all T tokens at the cost of one.
//   phase 1  routing-independent rows — router rows, the shared gate row and
//            the shared expert's gate/up pairs — as a CTA GEMV (B = the T x
//            rows in shared memory); logits are published in 16 copies,
//            shared activations in one.
//   phase 2  warp t gathers token t's logits and ranks them (lower index wins
//            ties) and forms its routing weights; every CTA then derives the
//            same union U of selected experts (ascending expert id) and the
//            weight of every (expert, token).
//   phase 3  the |U| * I gate/up pairs of the union, a contiguous range per
//            CTA, in passes of 8 pairs (gate rows on tile rows 0-7, the
//            matching up rows on 8-15); w * silu(gate) * up is published per
//            (pair, routed token).
//   phase 4  the down GEMV in units of 16 output rows of one expert, a
//            contiguous range of units per CTA: the CTA gathers the
//            activations of the experts its units touch, splits each into two
//            storage-type terms (B columns: token x term) and each warp runs
//            whole units; the weighted partial rows go out as exchange words.
//   The CTA's weight rows of phases 3 and 4 (the gate rows and the up rows of
//   each pass, then its W2 units) flow through one shared-memory ring of 1-D
//   bulk copies (mbarrier-tracked, refilled at every pass barrier), so the W2
//   rows land while the activations are exchanged.  Each bulk copy moves a
//   group of 2 consecutive rows and groups are padded by 16 bytes; the
//   tensor-core tiles take their rows in an order that puts the 8 rows of
//   every ldmatrix in 8 different bank groups (rows of different groups, and
//   gate and up rows from stages 64 bytes apart modulo 128), so the eight
//   warps' ldmatrix reads are free of bank conflicts.  x's B fragments stay
//   in registers for the whole of phase 3.
//   phase 5  CTA c sums, for its output rows and every token, the k routed
//            partials in slot order and the gated shared partial (plus x
//            with the residual flag) and writes out.
// Every exchange wait is bounded by the GPU global timer and records an error
// instead of hanging.  Programmatic dependent launch is triggered at entry.

#include <algorithm>
#include <type_traits>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kBtThreads = 256;             // the 8 computing warps
constexpr int kBtWarps = kBtThreads / 32;
constexpr int kBtBlock = kBtThreads + 32;   // plus the warp that issues the ring's copies
constexpr int kBtMaxPairs = kBatchMaxT * 8;  // T * k
constexpr int kBtRows1 = 32;     // routing-independent rows per CTA (host-checked)
constexpr int kBtMaxSlots = 4;   // activation slots one CTA's W2 units may touch (host-checked)
constexpr int kBtMaxStages = 8;  // ring stages
constexpr int kBtMaxCtas = 256;  // CTAs (flag words per activation slot)

namespace {

// 16-byte streaming weight load, or zeros without a load when `pred` is false.
// Volatile, so loads issued before griddepcontrol.wait stay there.
__device__ __forceinline__ uint4 ldg16_pred(const void* p, bool pred) {
  uint4 r;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\tmov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\t"
      "mov.b32 %3, 0;\n\t@q ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "r"(static_cast<int>(pred)));
  return r;
}

// 16-byte shared load, or zeros without a load when `pred` is false.
__device__ __forceinline__ uint4 lds16_pred(uint32_t addr, bool pred) {
  uint4 r;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\tmov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\t"
      "mov.b32 %3, 0;\n\t@q ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "r"(addr), "r"(static_cast<int>(pred)));
  return r;
}

// fp32 activation data exchanged with flags: plain stores by the producers,
// then a flag (the launch epoch) per (slot, producing CTA) after a CTA-wide
// barrier and a fence; consumers poll the flags, then read the data at GPU
// scope (not through L1).
__device__ __forceinline__ void st_flag(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ float4 ld_gpu_f4(const float* p) {
  float4 v;
  asm volatile("ld.relaxed.gpu.global.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Barrier of the 8 computing warps only (the copy-issuing warp never joins).
__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kBtThreads) : "memory"); }

// `n` arrivals on an mbarrier (one thread).
__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// One 16-row A tile of a warp's 256-column slice, held in registers: lane
// (g, t) keeps 16-byte chunks of rows g and g + 8 at columns c0 + 32 jj + 8 t
// (jj < 8).  Within a chunk, elements 0-3 form one m16n8k16 k-step and 4-7
// the next; B is read at the same columns, so the k order is the same on both
// sides.  B column n (= lane / 4) is row n of a shared-memory matrix of
// 2-byte elements, `bstride` bytes apart.
template <int DT>
struct TileGemv {
  uint4 w[2][8];

  __device__ __forceinline__ void load_global(const uint8_t* r0, bool v0, const uint8_t* r1, bool v1, int c0,
                                              int cend, int t) {
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int c = c0 + 32 * jj + 8 * t;
      const bool in = c < cend;
      const size_t off = 2 * static_cast<size_t>(in ? c : 0);
      w[0][jj] = ldg16_pred(r0 + off, in && v0);
      w[1][jj] = ldg16_pred(r1 + off, in && v1);
    }
  }

  __device__ __forceinline__ void load_shared(uint32_t r0, uint32_t r1, int c0, int cend, int t) {
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int c = c0 + 32 * jj + 8 * t;
      const bool in = c < cend;
      const uint32_t off = 2 * static_cast<uint32_t>(in ? c : 0);
      w[0][jj] = lds16_pred(r0 + off, in);
      w[1][jj] = lds16_pred(r1 + off, in);
    }
  }

  // acc (two alternating chains) += A x B over the slice, B columns n < nb.
  __device__ __forceinline__ void mma(uint32_t bbase, uint32_t bstride, int nb, int c0, int cend, int lane,
                                      float (&acc)[2][4]) const {
    const int n = lane >> 2, t = lane & 3;
    const bool bl = n < nb;
    const uint32_t brow = bbase + static_cast<uint32_t>(n) * bstride;
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
      const int c = c0 + 32 * jj + 8 * t;
      const bool in = c < cend;
      const uint4 b = lds16_pred(brow + 2 * static_cast<uint32_t>(in ? c : 0), bl && in);
      mma16816<DT>(acc[jj & 1], w[0][jj].x, w[1][jj].x, w[0][jj].y, w[1][jj].y, b.x, b.y);
      mma16816<DT>(acc[jj & 1], w[0][jj].z, w[1][jj].z, w[0][jj].w, w[1][jj].w, b.z, b.w);
    }
  }
};

// Lane (g, t) of a finished tile holds rows g / g + 8 of columns 2t, 2t + 1
// (columns c0 + 2t, c0 + 2t + 1 of part).
template <int W>
__device__ __forceinline__ void store_tile(float (*part)[W], int row0, int c0, int lane, const float (&acc)[2][4]) {
  const int g = lane >> 2, t = lane & 3;
  part[row0 + g][c0 + 2 * t] = acc[0][0] + acc[1][0];
  part[row0 + g][c0 + 2 * t + 1] = acc[0][1] + acc[1][1];
  part[row0 + g + 8][c0 + 2 * t] = acc[0][2] + acc[1][2];
  part[row0 + g + 8][c0 + 2 * t + 1] = acc[0][3] + acc[1][3];
}

// v ~ t0 + t1 in the storage type (t0 = rn(v), t1 = rn(v - t0)), packed
// pairwise: term[s] holds term s of v.x (low half) and v.y.
template <int DT>
__device__ __forceinline__ void split_terms(float2 v, uint32_t (&term)[2]) {
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

}  // namespace

struct BatchArgs {
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
  uint64_t* ll_logits;  // kLogitReplicas copies of [T][Lst] words, lrep words apart
  float* act;           // [(T*k + 1) slots][T][Imax] fp32 activations (slot T*k: shared expert)
  uint32_t* act_flag;   // [(T*k + 1) slots][kBtMaxCtas]: epoch once a CTA's share of the slot is out
  uint64_t* ll_part;    // [(T*k + 1) slots][T][H] words
  int T, H, E, k, I, Is, has_gate, norm_topk, out_dtype;
  int static_weights, residual;
  int Lst, lrep, Imax;
  uint32_t xs, cs;   // shared-memory strides (bytes): x rows, activation-term columns
  uint32_t gs13;     // ring: bytes between 2-row groups of W13 rows (2 H * 2 + 16)
  uint32_t gs2;      // ring: bytes between 2-row groups of a W2 unit (2 max(I, Is) * 2 + 16)
  uint32_t stage;    // ring stage bytes (8 W13 rows, or two W2 units of 16 rows), 64 modulo 128
  int ns;            // ring stages
  uint32_t off_terms, off_ring, off_xh, off_lg;  // x rows and logits (in the ring with x_in_ring)
  int x_in_ring;  // 1: the x rows and logits use the ring's space until its first copy
  uint64_t timeout_ns;
#ifdef MOE_PHASE_TRACE
  uint64_t* trace;  // this launch's record: [CTA][kTraceSlots]
#endif
};

// MAXT: the most tokens of the instantiation (8 or 16): the tokens are
// MAXT / 8 B-column blocks of the weight GEMVs and the two activation terms
// per token MAXT / 4 blocks of the down GEMV.
template <int DT, int MAXT>
__global__ void __launch_bounds__(kBtBlock, 1) decode_batch_kernel(const BatchArgs a) {
  constexpr int NBT = MAXT / 8, NBC = MAXT / 4, MAXP = MAXT * 8;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_red[kBtWarps][kBtRows1][MAXT];  // per-warp partial tiles (rows x tokens)
  __shared__ int s_ids[MAXT][8];
  __shared__ float s_sel[MAXT][8];
  __shared__ float s_w[MAXT][8];
  __shared__ float s_gate[MAXT];
  __shared__ float s_uw[MAXP][MAXT];      // routing weight of (union expert, token), 0 = not routed
  __shared__ uint32_t s_utok[MAXP];       // tokens routed to a union expert (bit t)
  __shared__ int s_uexp[MAXP];            // expert id of union slot u (ascending)
  __shared__ int s_uslot[MAXT][8];        // union slot of (token, rank)
  __shared__ float s_unsc[kBtMaxSlots][MAXT];  // fp16: the power of two undoing a row's term scale
  __shared__ __align__(8) uint64_t s_full[kBtMaxStages];   // ring stage landed
  __shared__ __align__(8) uint64_t s_empty[kBtMaxStages];  // ring stage read by the 8 computing warps
  __shared__ int s_nU;
  __shared__ uint32_t s_epoch, s_fail;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int cta = blockIdx.x, G = gridDim.x;
  const int T = a.T, H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is;
  const int E1 = E + a.has_gate;
  const int SH = T * k;  // exchange slot of the shared expert
  const size_t rowb = static_cast<size_t>(H) * 2;
  const int nch = H >> 3;
  uint8_t* xh = smem + a.off_xh;  // phase 1, and phase 3's B fragments
  uint8_t* ring = smem + a.off_ring;
  float* lg = reinterpret_cast<float*>(smem + a.off_lg);  // phase 2 only
  const uint32_t xha = smem_u32(xh);
  const uint32_t terms_a = smem_u32(smem + a.off_terms);
  const uint32_t ring_a = smem_u32(ring);
  const uint32_t stage_bytes = a.stage;
  constexpr int LREP = kLogitReplicas;

  MOE_STAMP(0);  // entry
  for (int i = tid; i < MAXP * MAXT; i += kBtThreads) (&s_uw[0][0])[i] = 0.0f;
  if (tid < MAXP) s_utok[tid] = 0u;
  if (tid == 0) {
    s_fail = 0;
    for (int st = 0; st < a.ns; ++st) {
      mbar_init(&s_full[st], 1);
      mbar_init(&s_empty[st], kBtWarps);
    }
    mbar_fence_init();
  }
  // x and the epoch word are read right after the PDL wait; start their DRAM
  // trips now (into L2 only, so the wait still orders the reads that count).
  for (int l = tid; l < (T * H * 2 + 127) >> 7; l += kBtThreads) prefetch_l2(a.x + 128 * static_cast<size_t>(l));
  if (tid == kBtThreads - 1) prefetch_l2(&a.ctrl->gen);
  pdl_launch_dependents();
  __syncthreads();  // the only barrier of all 288 threads

  // This CTA's work once the union U of selected experts is known (nU of
  // them): its gate/up pairs [pb0, pb1) of the |U| * I, in passes of 8, and
  // its W2 units [ub0, ub1) (16 output rows of one expert: union slot s < nU,
  // or the shared expert, s == nU).  Ring items: [0, n13) the W13 rows of the
  // passes (item 2 q: the gate rows of pass q's pairs, 2 q + 1: their up
  // rows, so a pass's two stages are adjacent: ns is even), then the W2 unit
  // pairs (item n13 + m: units ub0 + 2 m, + 1, 8 gs2 bytes apart).  Item i
  // uses stage i % ns, phase (i / ns) & 1.
  struct Plan {
    int pb0, pb1, npass, ub0, ub1, n13, nw2, nitems;
  };
  const int HB = H >> 4;
  const uint32_t rb13 = static_cast<uint32_t>(H) * 2;
  const uint32_t unit_bytes = 8u * a.gs2;
  auto make_plan = [&](int nU) -> Plan {
    Plan p;
    const int PU = nU * I;
    p.pb0 = static_cast<int>((static_cast<long long>(PU) * cta) / G);
    p.pb1 = static_cast<int>((static_cast<long long>(PU) * (cta + 1)) / G);
    p.npass = (p.pb1 - p.pb0 + 7) >> 3;
    const int NUn = nU > 0 ? (nU + (Is > 0 ? 1 : 0)) * HB : 0;
    p.ub0 = static_cast<int>((static_cast<long long>(NUn) * cta) / G);
    p.ub1 = static_cast<int>((static_cast<long long>(NUn) * (cta + 1)) / G);
    p.n13 = 2 * p.npass;
    p.nw2 = (p.ub1 - p.ub0 + 1) >> 1;
    p.nitems = p.n13 + p.nw2;
    return p;
  };
  auto unit_src = [&](int un, int nU, int& Iu) -> const uint8_t* {
    const int s = un / HB, hb = un - s * HB;
    if (s < nU) {
      Iu = I;
      return a.w2 + (static_cast<size_t>(s_uexp[s]) * H + hb * 16) * static_cast<size_t>(I) * 2;
    }
    Iu = Is;
    return a.sw2 + static_cast<size_t>(hb) * 16 * Is * 2;
  };

  if (warp == kBtWarps) {
    // ---- the copy-issuing warp.  A bulk copy stalls its warp while the
    // SM's copy queue is full, so no computing warp issues them: this warp
    // waits for the union, then streams the CTA's items into the ring, each
    // as soon as its stage has been read (s_empty), and lets every copy land
    // before it exits.  Every wait is bounded.
    pdl_wait();
    asm volatile("bar.sync 2, %0;" ::"r"(kBtBlock) : "memory");  // union formed
    const int nU = s_nU;
    const Plan pl = make_plan(nU);
    int issued = 0;
    for (; issued < pl.nitems; ++issued) {
      const int st = issued % a.ns;
      if (issued >= a.ns) {
        const bool ok = mbar_wait_until(&s_empty[st], ((issued / a.ns) - 1) & 1, global_ns() + a.timeout_ns);
        if (!__all_sync(0xffffffffu, ok)) break;  // the computing warps stopped
      }
      uint8_t* dst0 = ring + st * stage_bytes;
      uint32_t bytes = 0;
      const uint8_t* src[2] = {nullptr, nullptr};
      uint8_t* dst[2] = {nullptr, nullptr};
      uint32_t len[2] = {0, 0};
      if (issued < pl.n13) {
        // lane j < 4: tile rows 2j, 2j + 1 (pairs pbase + 2j, + 1), one copy
        // when both pairs are of the same expert (consecutive rows)
        const int q = issued >> 1, up = issued & 1;
        const int pbase = pl.pb0 + 8 * q;
        const int nv = min(8, pl.pb1 - pbase);
        bytes = static_cast<uint32_t>(nv) * rb13;
        const int r0 = 2 * lane;
        if (lane < 4 && r0 < nv) {
          auto row_of = [&](int p) -> const uint8_t* {
            const int u = p / I, i = p - u * I;
            return a.w13 + (static_cast<size_t>(s_uexp[u]) * 2 * I + (up ? I : 0) + i) * rb13;
          };
          const int pa = pbase + r0;
          const bool two = r0 + 1 < nv;
          const bool same = two && (pa / I == (pa + 1) / I);
          src[0] = row_of(pa);
          dst[0] = dst0 + lane * a.gs13;
          len[0] = same ? 2 * rb13 : rb13;
          if (two && !same) {
            src[1] = row_of(pa + 1);
            dst[1] = dst0 + lane * a.gs13 + rb13;
            len[1] = rb13;
          }
        }
      } else {
        // lane 8 v + j < 16: rows 2j, 2j + 1 of unit v of the pair
        const int m = issued - pl.n13;
#pragma unroll
        for (int v = 0; v < 2; ++v) {
          const int un = pl.ub0 + 2 * m + v;
          if (un < pl.ub1) {
            int Iu;
            const uint8_t* us = unit_src(un, nU, Iu);
            bytes += 16u * Iu * 2u;
            if ((lane >> 3) == v) {
              const int j = lane & 7;
              src[0] = us + static_cast<size_t>(2 * j) * Iu * 2;
              dst[0] = dst0 + v * unit_bytes + j * a.gs2;
              len[0] = 2u * Iu * 2u;
            }
          }
        }
      }
      if (lane == 0) mbar_arrive_expect_tx(&s_full[st], bytes);
      __syncwarp();
      if (src[0]) bulk_g2s(dst[0], src[0], len[0], &s_full[st]);
      if (src[1]) bulk_g2s(dst[1], src[1], len[1], &s_full[st]);
    }
    const uint64_t dl = global_ns() + a.timeout_ns;
    for (int it = max(0, issued - a.ns); it < issued; ++it) mbar_wait_until(&s_full[it % a.ns], (it / a.ns) & 1, dl);
    return;
  }

  // ---- phase 1: routing-independent rows of this CTA (router rows u = cta +
  // qG < E1, then its shared-expert pairs: gate rows, then up rows)
  const int n1 = E1 + Is;
  const int nL = cta < E1 ? (E1 - 1 - cta) / G + 1 : 0;
  const int nU1 = cta < n1 ? (n1 - 1 - cta) / G + 1 : 0;
  const int nS = nU1 - nL;
  const int R1 = nL + 2 * nS;
  auto p1_row = [&](int r, bool& valid) -> const uint8_t* {
    valid = r < R1;
    const int rr = r - nL;
    const int pi = rr < nS ? rr : rr - nS;
    const int uL = min(cta + r * G, E);
    const int i = max(0, cta + (nL + pi) * G - E1);
    if (!valid) return a.wr;
    if (r < nL) return uL < E ? a.wr + static_cast<size_t>(uL) * rowb : a.swg;
    return a.sw13 + static_cast<size_t>(rr < nS ? i : Is + i) * rowb;
  };
  const int cpw = H / kBtWarps;  // <= 256 columns per warp (H <= 2048, host-checked)
  const int c0w = warp * cpw, cendw = c0w + cpw;
  TileGemv<DT> gv;
  {
    bool va, vb;
    const uint8_t* ra = p1_row(g, va);
    const uint8_t* rb = p1_row(g + 8, vb);
    if (a.static_weights) gv.load_global(ra, va, rb, vb, c0w, cendw, t4);
    pdl_wait();  // x (and anything else an earlier kernel wrote) is visible from here
    MOE_STAMP(1);  // PDL wait released
    if (!a.static_weights) gv.load_global(ra, va, rb, vb, c0w, cendw, t4);
  }
  uint32_t gen_prev = 0;
  if (tid == 0) gen_prev = ld_relaxed_u32(&a.ctrl->gen);
  for (int c = tid; c < T * nch; c += kBtThreads) {
    const int tk = c / nch, cc = c - tk * nch;
    const uint4 raw = ld_ordered16(a.x + tk * rowb + 16 * static_cast<size_t>(cc));
    *reinterpret_cast<uint4*>(xh + static_cast<size_t>(tk) * a.xs + 16 * cc) = raw;
  }
  if (tid == 0) {
    const uint32_t ep = gen_prev + 1u;
    s_epoch = ep ? ep : 1u;
    // The T = 1 kernel's arrival counter of the next epoch's parity: the
    // launch that last used it has completed; clear it for the next launch.
    if (cta == 0) atomicExch(&a.ctrl->arrive[(s_epoch + 1u) & 1u], 0u);
  }
  cons_sync();
  const uint32_t epoch = s_epoch;
  MOE_STAMP(2);  // x staged

  for (int rg = 0; rg < R1; rg += 16) {
    if (rg > 0) {
      bool va, vb;
      const uint8_t* ra = p1_row(rg + g, va);
      const uint8_t* rb = p1_row(rg + 8 + g, vb);
      gv.load_global(ra, va, rb, vb, c0w, cendw, t4);
    }
#pragma unroll
    for (int nb = 0; nb < NBT; ++nb) {  // tokens 8 nb .. 8 nb + 7
      float acc[2][4] = {};
      gv.mma(xha + nb * 8 * a.xs, a.xs, T - 8 * nb, c0w, cendw, lane, acc);
      store_tile(s_red[warp], rg, 8 * nb, lane, acc);
    }
  }
  cons_sync();
  MOE_STAMP(3);  // phase-1 dot products summed
  {
    // logit words in LREP copies (every CTA reads all of them), shared
    // activations (unweighted; the gate scales the shared partial) once
    const int nlw = nL * T * LREP;
    for (int q = tid; q < nlw + nS * T; q += kBtThreads) {
      if (q < nlw) {
        const int o = q / (T * LREP), rem = q - o * T * LREP, tk = rem / LREP, rep = rem - tk * LREP;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kBtWarps; ++w) v += s_red[w][o][tk];
        ll_store(a.ll_logits + static_cast<size_t>(rep) * a.lrep + static_cast<size_t>(tk) * a.Lst + cta + o * G, v,
                 epoch);
      } else {
        const int q2 = q - nlw, pi = q2 / T, tk = q2 - pi * T;
        float gs = 0.0f, us = 0.0f;
#pragma unroll
        for (int w = 0; w < kBtWarps; ++w) {
          gs += s_red[w][nL + pi][tk];
          us += s_red[w][nL + nS + pi][tk];
        }
        const int i = cta + (nL + pi) * G - E1;
        a.act[static_cast<size_t>(SH * T + tk) * a.Imax + i] = silu_f(gs) * us;
      }
    }
  }

  MOE_STAMP(4);  // phase-1 results published

  // ---- phase 2: per token, its logits, top-k and routing weights (warp t
  // takes tokens t, t + 8)
  for (int tw = warp; tw < T; tw += kBtWarps) {
    float* lw = lg + tw * a.Lst;
    const uint64_t* src = a.ll_logits + static_cast<size_t>(cta % LREP) * a.lrep + static_cast<size_t>(tw) * a.Lst;
    const bool ok = __all_sync(0xffffffffu, ll_gather<8>(src, lw, E1, lane, 32, epoch, global_ns() + a.timeout_ns));
    MOE_STAMP(5);  // logits gathered (warp 0)
    if (!ok) {
      if (lane == 0) s_fail = kDevTimeoutLogits;
    } else {
      warp_topk_sorted8(lw, E, k, s_ids[tw], s_sel[tw]);
      MOE_STAMP(15);  // warp 0's top-k done
      warp_routing_weights(lw, E, s_sel[tw], k, a.norm_topk, s_w[tw]);
      if (lane == 0) s_gate[tw] = a.has_gate ? sigmoid_f(lw[E]) : 1.0f;
      __syncwarp();
      if (cta == 0 && lane < k) {
        a.topk_ids[tw * k + lane] = s_ids[tw][lane];
        a.topk_w[tw * k + lane] = s_w[tw][lane];
      }
    }
  }
  cons_sync();
  MOE_STAMP(16);  // every token ranked
  const bool ranked = s_fail == 0;  // uniform: read after the barrier
  // Every CTA owns a logit row (G <= E + has_gate) and read the epoch before
  // publishing it; CTA 0 has now seen all of them, so the next launch may use
  // the next epoch.  The shared activations of phase 1 are out: flag them.
  // (the GPU-scope fence is slow: the last warp takes it, off warp 0's path)
  if (cta == 0 && tid == 0) atomicExch(&a.ctrl->gen, epoch);
  if (tid == kBtThreads - 32 && nS > 0) {
    __threadfence();
    st_flag(a.act_flag + static_cast<size_t>(SH) * kBtMaxCtas + cta, epoch);
  }
  if (ranked && warp == 0) {
    // the union U of selected experts (ascending id) and, per (token, rank),
    // its slot in U: lane l takes selections l, l + 32, ...; lane w < 8
    // keeps word w of the 256-bit selection mask (every loop is unrolled, so
    // nothing is indexed at run time: that would put the arrays in local
    // memory)
    constexpr int NSEL = MAXP / 32;
    int esel[NSEL];
#pragma unroll
    for (int h = 0; h < NSEL; ++h) {
      const int q = lane + 32 * h;
      esel[h] = q < T * k ? s_ids[q / k][q % k] : -1;
    }
    uint32_t word = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      uint32_t mine = 0;
#pragma unroll
      for (int h = 0; h < NSEL; ++h) mine |= esel[h] >= 0 && (esel[h] >> 5) == w ? 1u << (esel[h] & 31) : 0u;
      const uint32_t m = __reduce_or_sync(0xffffffffu, mine);
      if (lane == w) word = m;
    }
    const int cnt = __popc(word);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int excl = incl - cnt;
#pragma unroll
    for (int h = 0; h < NSEL; ++h) {
      const int q = lane + 32 * h, e = esel[h];
      const uint32_t mwd = __shfl_sync(0xffffffffu, word, max(e, 0) >> 5);
      const int base = __shfl_sync(0xffffffffu, excl, max(e, 0) >> 5);
      if (e >= 0) {
        const int u = base + __popc(mwd & ((1u << (e & 31)) - 1u));
        const int tk = q / k, j = q - tk * k;
        s_uslot[tk][j] = u;
        s_uw[u][tk] = s_w[tk][j];
        atomicOr(&s_utok[u], 1u << tk);
      }
    }
    if (lane < 8) {
      int r = excl;
      for (uint32_t mm = word; mm; mm &= mm - 1u) s_uexp[r++] = lane * 32 + __ffs(mm) - 1;
    }
    if (lane == 7) s_nU = incl;
    MOE_STAMP(17);  // warp 0: union formed
  }
  cons_sync();
  const int nU = ranked ? s_nU : 0;
  if (tid == 0) s_nU = nU;  // 0 when ranking failed: the copy-issuing warp then has nothing to do
  auto start_copies = [&]() { asm volatile("bar.arrive 2, %0;" ::"r"(kBtBlock) : "memory"); };
  if (!a.x_in_ring) start_copies();
  const Plan pl = make_plan(nU);
  const int pb0 = pl.pb0, pb1 = pl.pb1, npass = pl.npass, ub0 = pl.ub0, ub1 = pl.ub1, n13 = pl.n13, nw2 = pl.nw2;
  const int kpw = H >> 7;  // 16-column steps per warp (H / 8 columns each)
  // x's B fragments for this warp's 16-column steps of phase 3 (column n =
  // token g, rows k = 2t, 2t + 1 and 2t + 8, 2t + 9 of the step), read before
  // the ring's first copy overwrites the x rows
  uint32_t bx[NBT][16][2];
  auto load_bx = [&]() {
#pragma unroll
    for (int nb = 0; nb < NBT; ++nb)
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const int tk = 8 * nb + g;
        const bool in = npass > 0 && kk < kpw && tk < T;
        const int k0 = (warp * kpw + kk) * 16 + 2 * t4;
        const uint32_t xa = xha + static_cast<uint32_t>(in ? tk : 0) * a.xs + 2 * (in ? k0 : 0);
        bx[nb][kk][0] = in ? lds32(xa) : 0u;
        bx[nb][kk][1] = in ? lds32(xa + 16) : 0u;
      }
  };
  load_bx();
  if (a.x_in_ring) {
    cons_sync();  // every x read is done before the ring's first copy
    start_copies();
  }
  MOE_STAMP(6);  // ranked, union formed

  // ---- phase 3: this CTA's range of the union's gate/up pairs
  auto wait_item = [&](int it) {  // every computing thread; bounded
    if (!mbar_wait_until(&s_full[it % a.ns], (it / a.ns) & 1, global_ns() + a.timeout_ns)) s_fail = kDevTimeoutCopy;
  };
  auto release_item = [&](int it, uint32_t n) {  // this warp is done reading the item's stage
    __syncwarp();
    if (lane == 0) mbar_arrive_cnt(&s_empty[it % a.ns], n);
  };
  // tile rows: 0-3 gate rows of pairs 0, 2, 4, 6 of the pass, 4-7 their up
  // rows, 8-15 the same for pairs 1, 3, 5, 7
  auto publish_pass = [&](int q) {
    const int b = (q & 1) * 16;
    if (tid < 8 * T) {
      const int pg = tid / T, tk = tid - pg * T;
      const int p = pb0 + 8 * q + pg;
      const int rg = b + (pg & 1) * 8 + (pg >> 1);  // tile row of the pair's gate row (+4: up row)
      if (p < pb1) {
        const int u = p / I, i = p - u * I;
        if ((s_utok[u] >> tk) & 1u) {
          float gs = 0.0f, us = 0.0f;
#pragma unroll
          for (int w = 0; w < kBtWarps; ++w) {
            gs += s_red[w][rg][tk];
            us += s_red[w][rg + 4][tk];
          }
          a.act[static_cast<size_t>(u * T + tk) * a.Imax + i] = silu_f(gs) * us * s_uw[u][tk];
        }
      }
    }
  };
  // ldmatrix.x4 lane addresses (k 0-7 for lanes 0-15, k 8-15 for 16-31):
  // tile row (lane & 15) is row ((lane >> 3) & 1) of group (lane & 3) of the
  // gate item (lane & 4 clear) or of the up item
  const uint32_t lm13 = static_cast<uint32_t>(lane & 3) * a.gs13 + ((lane >> 3) & 1) * rb13 + (lane >> 4) * 16;
  if (npass > 0) {
    for (int q = 0; q < npass; ++q) {
      float acc[NBT][2][4] = {};
      wait_item(2 * q);
      wait_item(2 * q + 1);
      const uint32_t sa = ring_a + ((2 * q + ((lane >> 2) & 1)) % a.ns) * stage_bytes + lm13 +
                          static_cast<uint32_t>(warp * kpw) * 32;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        if (kk < kpw) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(sa + kk * 32, a0, a1, a2, a3);
#pragma unroll
          for (int nb = 0; nb < NBT; ++nb)
            mma16816<DT>(acc[nb][kk & 1], a0, a1, a2, a3, bx[nb][kk][0], bx[nb][kk][1]);
        }
      release_item(2 * q, 1);
      release_item(2 * q + 1, 1);
#pragma unroll
      for (int nb = 0; nb < NBT; ++nb) store_tile(s_red[warp], (q & 1) * 16, 8 * nb, lane, acc[nb]);
      if (q == 0) MOE_STAMP(12);  // thread 0: first pass's dot products done
      cons_sync();  // this pass's partials are visible
      if (q == 1) MOE_STAMP(13);  // second pass done (all warps)
      if (q == 2) MOE_STAMP(14);  // third pass done (all warps)
      publish_pass(q);
    }
  }
  if (npass > 0) {
    cons_sync();  // every activation of this CTA's pairs is stored
    if (tid == kBtThreads - 32) {  // the last warp: warps 0..nsl-1 poll flags next
      __threadfence();
      for (int s = pb0 / I; s <= (pb1 - 1) / I; ++s) st_flag(a.act_flag + static_cast<size_t>(s) * kBtMaxCtas + cta, epoch);
    }
  }
  MOE_STAMP(7);  // phase-3 passes done

  // ---- phase 4: activations of the slots this CTA's units touch, then the
  // units.  Warp ls < nsl waits for the flags of every CTA that produces
  // part of local slot ls (the CTAs whose pair range meets the slot; for the
  // shared expert, those with shared pairs); then each warp turns rows
  // (slot, token) into the two terms: a routed slot's routed tokens (the
  // others are zero), all T for the shared slot.
  const int s_lo = ub0 / HB;
  const int nsl = ub1 > ub0 ? (ub1 - 1) / HB - s_lo + 1 : 0;  // <= kBtMaxSlots (host-checked)
  const uint32_t slot_bytes = 2u * T * a.cs;
  if (ranked && warp < nsl) {
    const int s = s_lo + warp;
    const bool sh = s == nU;
    const int PU = nU * I;
    const uint32_t* fl = a.act_flag + static_cast<size_t>(sh ? SH : s) * kBtMaxCtas;
    const uint64_t dl = global_ns() + a.timeout_ns;
    bool ok = true;
    for (int c = lane; c < G; c += 32) {
      bool prod;
      if (sh) {
        const int n1c = E1 + Is;
        const int nLc = c < E1 ? (E1 - 1 - c) / G + 1 : 0, nUc = c < n1c ? (n1c - 1 - c) / G + 1 : 0;
        prod = nUc > nLc;
      } else {
        const int q0 = static_cast<int>((static_cast<long long>(PU) * c) / G);
        const int q1 = static_cast<int>((static_cast<long long>(PU) * (c + 1)) / G);
        prod = q1 > q0 && q0 < (s + 1) * I && q1 > s * I;
      }
      if (prod)
        while (ld_relaxed_u32(fl + c) != epoch)
          if (global_ns() > dl) {
            ok = false;
            break;
          }
    }
    if (!__all_sync(0xffffffffu, ok) && lane == 0) s_fail = kDevTimeoutAct;
  }
  cons_sync();  // the flags are in (or a wait ran out)
  MOE_STAMP(8);  // activations published (flags in)
  const bool have_act = ranked && s_fail == 0;
  if (have_act) {
    for (int row = warp; row < nsl * T; row += kBtWarps) {
      const int ls = row / T, tk = row - ls * T, s = s_lo + ls;
      const bool sh = s == nU;
      const int Iu = sh ? Is : I;
      const bool routed = sh || ((s_utok[s] >> tk) & 1u);
      const float* src = a.act + static_cast<size_t>((sh ? SH : s) * T + tk) * a.Imax;
      uint8_t* col = smem + a.off_terms + ls * slot_bytes + static_cast<size_t>(2 * tk) * a.cs;
      // terms: slot ls, column 2 * token + term, element i at
      // terms + ls * slot_bytes + column * cs + 2 i
      float sc = 1.0f, unsc = 1.0f;
      if constexpr (DT == MOE_F16) {
        // a power of two putting the row's largest magnitude in [2^14, 2^15)
        // (exact; undone on the unit's sums)
        float mx = 0.0f;
        for (int i = 4 * lane; i < Iu && routed; i += 128) {
          const float4 v = ld_gpu_f4(src + i);
          mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(mx));
        int shf = amax ? 14 - (static_cast<int>(amax >> 23) - 127) : 0;
        shf = max(-100, min(100, shf));
        sc = __int_as_float((127 + shf) << 23);
        unsc = __int_as_float((127 - shf) << 23);
      }
      if (lane == 0) s_unsc[ls][tk] = unsc;
      for (int i = 4 * lane; i < a.Imax; i += 128) {
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (routed && i < Iu) v = ld_gpu_f4(src + i);
        uint32_t t0[2], t1[2];
        split_terms<DT>(make_float2(v.x * sc, v.y * sc), t0);
        split_terms<DT>(make_float2(v.z * sc, v.w * sc), t1);
        *reinterpret_cast<uint2*>(col + 2 * i) = make_uint2(t0[0], t1[0]);
        *reinterpret_cast<uint2*>(col + a.cs + 2 * i) = make_uint2(t0[1], t1[1]);
      }
    }
  }
  cons_sync();
  MOE_STAMP(9);  // terms written
  // units: warp w runs unit slots w, w + 8, ... (item n13 + slot / 2); every
  // item is waited for and released, also when there is nothing to compute
  for (int us = warp; us < 2 * nw2; us += kBtWarps) {
    const int m = us >> 1, v = us & 1;
    const int un = ub0 + 2 * m + v;
    wait_item(n13 + m);
    if (us == 0) MOE_STAMP(18);  // warp 0's first unit landed
    if (have_act && un < ub1) {
      const int s = un / HB, hb = un - s * HB, ls = s - s_lo;
      const bool sh = s == nU;
      const int Iu = sh ? Is : I;
      // ldmatrix.x4 lane addresses: tile row (lane & 15) is unit row
      // 2 (lane & 7) + ((lane >> 3) & 1), the first or second row of group
      // (lane & 7); k 0-7 for lanes 0-15, 8-15 for 16-31
      const uint32_t sa = ring_a + ((n13 + m) % a.ns) * stage_bytes + v * unit_bytes +
                          static_cast<uint32_t>(lane & 7) * a.gs2 + ((lane >> 3) & 1) * Iu * 2 + (lane >> 4) * 16;
      const uint32_t bb = terms_a + ls * slot_bytes + static_cast<uint32_t>(g) * a.cs + 4 * t4;
      // B column block nc holds columns 8 nc .. 8 nc + 7 (tokens 4 nc .. 4 nc + 3)
      float acc[NBC][4][4] = {};
      // NK 16-column steps at a time: every operand load issued before the
      // tensor-core steps, four accumulator chains (static indices: a runtime
      // index would put the accumulators in local memory)
      auto ksteps = [&](auto nk_c, int ks) {
        constexpr int NK = decltype(nk_c)::value;
        uint32_t av[NK][4], xv[NK][NBC][2];
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          ldsm_x4(sa + (ks + i) * 32, av[i][0], av[i][1], av[i][2], av[i][3]);
          const uint32_t ba = bb + (ks + i) * 32;
#pragma unroll
          for (int nc = 0; nc < NBC; ++nc) {
            const bool bv = 8 * nc + g < 2 * T;
            xv[i][nc][0] = bv ? lds32(ba + 8 * nc * a.cs) : 0u;
            xv[i][nc][1] = bv ? lds32(ba + 8 * nc * a.cs + 16) : 0u;
          }
        }
#pragma unroll
        for (int i = 0; i < NK; ++i)
#pragma unroll
          for (int nc = 0; nc < NBC; ++nc)
            if (8 * nc < 2 * T)
              mma16816<DT>(acc[nc][i & 3], av[i][0], av[i][1], av[i][2], av[i][3], xv[i][nc][0], xv[i][nc][1]);
      };
      const int nks = Iu >> 4;
      int ks = 0;
      for (; ks + 4 <= nks; ks += 4) ksteps(std::integral_constant<int, 4>{}, ks);
      for (; ks < nks; ++ks) ksteps(std::integral_constant<int, 1>{}, ks);
      release_item(n13 + m, kBtWarps / 2);
      if (us == 0) MOE_STAMP(19);  // warp 0's first unit computed
      // lane (g, t4): tile rows g, g + 8 (unit rows 2g, 2g + 1) of tokens
      // 4 nc + t4 (columns hi, lo of block nc)
      auto publish = [&](int tk, const float(&ac)[4][4]) {
        if (tk < T && (sh || ((s_utok[s] >> tk) & 1u))) {
          float unsc = 1.0f;
          if constexpr (DT == MOE_F16) unsc = s_unsc[ls][tk];
          const float y0 = (((ac[0][0] + ac[1][0]) + (ac[2][0] + ac[3][0])) + ((ac[0][1] + ac[1][1]) + (ac[2][1] + ac[3][1]))) * unsc;
          const float y1 = (((ac[0][2] + ac[1][2]) + (ac[2][2] + ac[3][2])) + ((ac[0][3] + ac[1][3]) + (ac[2][3] + ac[3][3]))) * unsc;
          uint64_t* pr = a.ll_part + static_cast<size_t>((sh ? SH : s) * T + tk) * H + hb * 16;
          ll_store(pr + 2 * g, y0, epoch);
          ll_store(pr + 2 * g + 1, y1, epoch);
        }
      };
#pragma unroll
      for (int nc = 0; nc < NBC; ++nc) publish(4 * nc + t4, acc[nc]);
    } else {
      release_item(n13 + m, kBtWarps / 2);
    }
  }
  MOE_STAMP(10);  // warp 0's units done

  // ---- phase 5: this CTA's output rows for every token
  if (have_act) {
    const int h0 = static_cast<int>((static_cast<long long>(H) * cta) / G);
    const int hn = static_cast<int>((static_cast<long long>(H) * (cta + 1)) / G) - h0;
    for (int q = tid; q < T * hn; q += kBtThreads) {
      const int tk = q / hn, h = h0 + (q - tk * hn);
      uint64_t wv[9];
      uint32_t want = 0;
#pragma unroll
      for (int j = 0; j < 9; ++j) {
        const bool in = j < k || (j == 8 && Is > 0);
        const int S = j < k ? s_uslot[tk][j] : SH;
        wv[j] = ll_load1_pred(a.ll_part + static_cast<size_t>(S * T + tk) * H + h, in);
        want |= (in ? 1u : 0u) << j;
      }
      const uint64_t dl = global_ns() + a.timeout_ns;
      bool ok = true;
      for (;;) {
        uint32_t missing = 0;
#pragma unroll
        for (int j = 0; j < 9; ++j)
          if (((want >> j) & 1u) && static_cast<uint32_t>(wv[j] >> 32) != epoch) missing |= 1u << j;
        if (!missing) break;
        if (global_ns() > dl) {
          ok = false;
          break;
        }
#pragma unroll
        for (int j = 0; j < 9; ++j) {
          const bool re = (missing >> j) & 1u;
          const int S = j < k ? s_uslot[tk][j] : SH;
          if (re) wv[j] = ll_load1_pred(a.ll_part + static_cast<size_t>(S * T + tk) * H + h, true);
        }
      }
      if (!ok) {
        s_fail = kDevTimeoutAct;
        continue;
      }
      float sum = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < k) sum += __uint_as_float(static_cast<uint32_t>(wv[j]));
      if (Is > 0) sum += s_gate[tk] * __uint_as_float(static_cast<uint32_t>(wv[8]));
      if (a.residual) sum += load_scalar<DT>(a.x + static_cast<size_t>(tk) * rowb, h);  // x, exact in fp32
      store_out(a.out, static_cast<size_t>(tk) * H + h, sum, a.out_dtype);
    }
  }
  MOE_STAMP(11);  // thread 0's outputs written
  cons_sync();
  if (tid == 0 && s_fail) report_error(a.ctrl, s_fail, static_cast<uint32_t>(cta));
}

// ------------------------------------------------------------------ host side
namespace {

struct BatchGeom {
  int G = 0, Lst = 0, Imax = 0, ns = 0;
  uint32_t xs = 0, cs = 0, gs13 = 0, gs2 = 0, stage = 0;
  uint32_t off_terms = 0, off_ring = 0, off_xh = 0, off_lg = 0;
  bool x_in_ring = false;
  size_t smem = 0;  // dynamic shared memory per CTA
  int nsl = 0;      // activation slots one CTA's units may touch
};

// Static shared memory of decode_batch_kernel (the arrays declared in it,
// for at most 8 and at most 16 tokens), rounded up; the dynamic part gets the
// rest of the 227 KB.
static size_t bt_static_smem(int32_t T) { return T <= 8 ? 16 * 1024 : 32 * 1024; }

BatchGeom batch_geom(const moe_cfg_t& c, int32_t T) {
  BatchGeom b;
  const int H = c.hidden, E1 = c.n_experts + c.has_shared_gate, k = c.top_k;
  const int Imax = c.inter > c.shared_inter ? c.inter : c.shared_inter;
  b.G = sm_count() < E1 ? sm_count() : E1;
  b.Lst = (E1 + 1) & ~1;
  b.Imax = Imax;
  // x rows 64 bytes past a multiple of 128 (the 16-byte B loads of lanes
  // (g, t) and (g + 1, t) fall in different bank halves); term columns 16
  // bytes past (8 columns hit 8 different bank groups)
  b.xs = static_cast<uint32_t>(align_up(static_cast<size_t>(H) * 2, 128) + 64);
  b.cs = static_cast<uint32_t>(align_up(static_cast<size_t>(Imax) * 2, 128) + 16);
  // ring: rows in 2-row groups, each followed by 16 bytes of padding
  b.gs13 = static_cast<uint32_t>(2 * H * 2 + 16);
  b.gs2 = static_cast<uint32_t>(2 * Imax * 2 + 16);
  b.stage = static_cast<uint32_t>(align_up(std::max(4u * b.gs13, 2u * 8u * b.gs2), 128) + 64);
  const int HB = H / 16;
  const long long nun_max = static_cast<long long>(T * k + (c.shared_inter > 0 ? 1 : 0)) * HB;
  const int upc = static_cast<int>((nun_max + b.G - 1) / b.G);  // units per CTA, at most
  b.nsl = upc > 0 ? (upc - 1) / HB + 2 : 0;
  // [x rows][activation terms][ring], or, when that gains a ring stage,
  // [activation terms][ring] with the x rows and then the logits in the
  // ring's space until its first copy (a barrier before the first copy then
  // keeps the x reads ahead of it)
  const size_t xbytes = align_up(static_cast<size_t>(T) * b.xs, 128);
  const size_t tbytes = align_up(static_cast<size_t>(b.nsl) * 2 * T * b.cs, 128);
  {
    const size_t bud = 227 * 1024 - bt_static_smem(T);
    const size_t sep = xbytes + tbytes < bud ? (bud - xbytes - tbytes) / b.stage : 0;
    const size_t ali = tbytes < bud ? (bud - tbytes) / b.stage : 0;
    b.x_in_ring = std::min<size_t>(ali, kBtMaxStages) > std::min<size_t>(sep, kBtMaxStages);
  }
  size_t off = 0;
  if (!b.x_in_ring) {
    b.off_xh = 0;
    off += xbytes;
  }
  b.off_terms = static_cast<uint32_t>(off);
  off += align_up(static_cast<size_t>(b.nsl) * 2 * T * b.cs, 128);
  b.off_ring = static_cast<uint32_t>(off);
  if (b.x_in_ring) b.off_xh = b.off_ring;
  b.off_lg = static_cast<uint32_t>(b.x_in_ring ? off + xbytes : off);
  const size_t budget = 227 * 1024 - bt_static_smem(T);
  const size_t ns = off < budget ? (budget - off) / b.stage : 0;
  // an even count keeps every pass's gate and up stages adjacent (64 bytes
  // apart modulo 128); an odd one costs 2-way conflicts on the wrapping pass
  b.ns = static_cast<int>(ns > static_cast<size_t>(kBtMaxStages) ? kBtMaxStages : ns);
  const size_t ring = std::max(static_cast<size_t>(b.ns) * b.stage,
                               (b.x_in_ring ? xbytes : 0) + static_cast<size_t>(T) * b.Lst * 4);
  b.smem = off + ring;
  return b;
}

}  // namespace

bool batch_ws_shape_ok(const moe_cfg_t& c, int32_t T) {
  if (T < 2 || T > kBatchMaxT) return false;
  const int H = c.hidden, E = c.n_experts, k = c.top_k, I = c.inter, Is = c.shared_inter;
  if (E > 256 || k > 8 || T * k > kBtMaxPairs) return false;
  if (H % 256 != 0 || H > 2048) return false;  // whole 16-column steps per warp and segment
  return I % 16 == 0 && Is % 16 == 0;
}

bool batch_shape_ok(const moe_cfg_t& c, int32_t T) {
  if (!batch_ws_shape_ok(c, T)) return false;
  const int E1 = c.n_experts + c.has_shared_gate, Is = c.shared_inter;
  const BatchGeom b = batch_geom(c, T);
  if (b.G < 1 || b.G > E1 || b.G > kBtMaxCtas) return false;  // every CTA owns a logit row
  if (2 * ((E1 + Is + b.G - 1) / b.G) > kBtRows1) return false;
  if (b.nsl > kBtMaxSlots) return false;
  return b.ns >= 2;
}

static size_t batch_act_data_bytes(const moe_cfg_t& c, int32_t T) {
  const int Imax = c.inter > c.shared_inter ? c.inter : c.shared_inter;
  return align_up((static_cast<size_t>(T) * c.top_k + 1) * T * Imax * 4, kWsAlign);
}

size_t batch_ws_words(const moe_cfg_t& c, int32_t T, size_t& logit_words, size_t& act_words) {
  const int E1 = c.n_experts + c.has_shared_gate;
  const size_t slots = static_cast<size_t>(T) * c.top_k + 1;
  logit_words = static_cast<size_t>(kLogitReplicas) * T * ((E1 + 1) & ~1);
  // fp32 activations, then one flag word per (slot, CTA)
  act_words = (batch_act_data_bytes(c, T) + slots * kBtMaxCtas * 4 + 7) / 8;
  return slots * T * c.hidden;  // partial words
}

moe_status_t launch_decode_batch(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws, const WsLayout& L,
                                 int32_t T, cudaStream_t st) {
  if (!batch_shape_ok(c, T) || !L.bt_logits)
    return set_error(MOE_ERR_UNSUPPORTED, "single-launch batch path: needs 2 <= T <= 16, E <= 256, k <= 8, "
                                          "H a multiple of 256 up to 2048, I and Is multiples of 16");
  const BatchGeom b = batch_geom(c, T);
  BatchArgs a;
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
  a.ll_logits = reinterpret_cast<uint64_t*>(ws + L.bt_logits);
  a.act = reinterpret_cast<float*>(ws + L.bt_act);
  a.act_flag = reinterpret_cast<uint32_t*>(ws + L.bt_act + batch_act_data_bytes(c, T));
  a.ll_part = reinterpret_cast<uint64_t*>(ws + L.bt_part);
  a.T = T;
  a.H = c.hidden; a.E = c.n_experts; a.k = c.top_k; a.I = c.inter; a.Is = c.shared_inter;
  a.has_gate = c.has_shared_gate; a.norm_topk = c.norm_topk; a.out_dtype = c.out_dtype;
  a.static_weights = (c.flags & MOE_FLAG_STATIC_WEIGHTS) ? 1 : 0;
  a.residual = (c.flags & MOE_FLAG_RESIDUAL) ? 1 : 0;
  a.Lst = b.Lst;
  a.lrep = T * b.Lst;
  a.Imax = b.Imax;
  a.xs = b.xs; a.cs = b.cs;
  a.gs13 = b.gs13; a.gs2 = b.gs2; a.stage = b.stage; a.ns = b.ns;
  a.off_terms = b.off_terms; a.off_ring = b.off_ring; a.off_xh = b.off_xh; a.off_lg = b.off_lg;
  a.x_in_ring = b.x_in_ring ? 1 : 0;
  a.timeout_ns = wait_timeout_ns();
#ifdef MOE_PHASE_TRACE
  a.trace = trace_next_record();
  if (!a.trace) return check_launch("trace buffer");
  if (b.G > kTraceCtas) return set_error(MOE_ERR_UNSUPPORTED, "trace build: more than %d CTAs", kTraceCtas);
#endif
  const size_t smem = b.smem;

  auto launch = [&](auto kernel) -> moe_status_t {
    if (raise_smem_limit(kernel, smem) != cudaSuccess) return check_launch("cudaFuncSetAttribute(batch)");
    // CTAs wait for one another's words: all G must be resident at once.
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBtBlock, smem) != cudaSuccess) {
      cudaGetLastError();
      return set_error(MOE_ERR_CUDA, "batch: occupancy query failed");
    }
    if (static_cast<long long>(per_sm) * sm_count() < b.G)
      return set_error(MOE_ERR_UNSUPPORTED, "batch: %d CTAs must be co-resident, %d per SM fit", b.G, per_sm);
    if (launch_pdl(kernel, dim3(b.G), dim3(kBtBlock), smem, st, a) != cudaSuccess)
      return check_launch("decode_batch_kernel");
    stat_kernels(1);
    return MOE_OK;
  };
  if (T <= 8) {
    if (c.dtype == MOE_BF16) return launch(decode_batch_kernel<MOE_BF16, 8>);
    return launch(decode_batch_kernel<MOE_F16, 8>);
  }
  if (c.dtype == MOE_BF16) return launch(decode_batch_kernel<MOE_BF16, 16>);
  return launch(decode_batch_kernel<MOE_F16, 16>);
}

}  // namespace moe
