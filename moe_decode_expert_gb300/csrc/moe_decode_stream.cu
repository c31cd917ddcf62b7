// moe_decode_stream.cu — the T = 1 decode MoE block in one launch, every
// weight byte streamed by TMA, the down projection split by columns.
//
// What it computes ("BI-V100 inference work log", Parts 3, 4, 9, 10): the same
// block as moe_decode.cu — router GEMV, softmax and top-k, the direct-routed
// W13 GEMV W13[expert_ids[k], row, :] with SiluAndMul, the W2 GEMV
// W2[expert_ids[k], h, :] weighted by the routing weights, and the shared
// expert with its optional sigmoid gate.
//
// How (GB300 design; the standard shapes — E <= 256, k <= 8, I and Is
// multiples of 16, H a multiple of 256 up to 4096 — all other shapes run the
// kernel of moe_decode.cu):
//  * The k*I routed and Is shared activation columns form units of 16
//    columns.  Units go round-robin to clusters of two CTAs.  CTA rank s of a
//    cluster computes the gate/up dot products of columns 8s..8s+7 of the unit
//    (16 W13 rows), writes its 8 activations into its partner's shared memory
//    as well, and, with all 16, runs the unit's down projection for output
//    rows [s*H/2, (s+1)*H/2): H/2 W2 rows x 16 columns, added to the CTA's
//    partial output.  Every weight byte is read once, by one CTA.
//  * Weights move by TMA into a ring of NS stages of 16*H bytes, tracked by
//    mbarriers and filled by a producer warp: a W13 stage is 16 row halves
//    (one bulk copy each, into rows padded by 16 bytes so ldmatrix is
//    conflict-free), a W2 stage is H/2 rows x 16 columns in tiled copies
//    through a 2-D tensor map.  Eight consumer warps run m16n8k16 steps on
//    each stage: W13 rows as A with x as column 0 of B; W2 rows as A with the
//    16 activations, split into three storage-type terms, as columns 0-2 of B.
//  * The shared expert's units do not depend on the routing: their stages go
//    out at entry (before the PDL wait with static weights).  Routed stages go
//    out as soon as this CTA has ranked the logits.
//  * Routing: every CTA computes ceil((E+1)/G) router rows (row E: the shared
//    gate vector) from registers loaded at entry, publishes them as
//    (value, epoch) words, gathers all of them and ranks them itself (fp32,
//    lower index first on ties): no grid barrier.
//  * Output: each CTA publishes its partial output rows as (value, epoch)
//    words, then sums, for its own H/G output rows, the partials of every
//    cluster in cluster order (deterministic), adds x when the residual flag
//    is set, and writes out.
// Every wait is bounded by the GPU global timer and records an error instead
// of hanging; the copies a CTA has in flight are waited for (bounded) and the
// pair meets at a cluster barrier before either exits, so no copy or remote
// store lands in shared memory that has been handed to another CTA.

#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

constexpr int kStrCons = 8;                       // consumer warps
constexpr int kStrThreads = 32 * (kStrCons + 1);  // + the producer warp
constexpr int kStrMaxUnits = 8;                   // units per cluster
constexpr int kStrMaxRouterRows = 4;              // router rows per CTA
constexpr int kStrMaxStages = 6;                  // ring stages
constexpr int kStrMaxMt = 16;                     // m-tiles per warp in a W2 stage (H <= 4096)
constexpr int kStrGather = 8;                     // partial words per thread in the final sum

struct StreamArgs {
  const uint8_t* x;
  const uint8_t* wr;
  const uint8_t* w13;
  const uint8_t* sw13;
  const uint8_t* swg;
  int32_t* topk_ids;
  float* topk_w;
  void* out;
  Control* ctrl;
  uint64_t* ll_logits;  // kLogitReplicas copies, ll_stride words apart
  uint64_t* ll_part;    // partial-output words [C][H]
  int H, E, k, I, Is, has_gate, norm_topk, out_dtype, static_weights, residual;
  int ll_stride;
  int C, U, Us;          // clusters, units, shared units (unit ids 0..Us-1)
  int NS;                // ring stages
  int box_rows;          // W2 rows per tiled copy
  uint32_t pitch;        // shared-memory pitch of a W13 row half: H + 16 bytes
  uint32_t stage_bytes;  // ring stage size
  uint32_t off_x, off_lg, off_act, off_red;
  uint64_t timeout_ns;
#ifdef MOE_PHASE_TRACE
  uint64_t* trace;
#endif
};

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
// The address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Arrive on an mbarrier of another CTA of the cluster, releasing this thread's
// earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
}
// try_wait with acquire at cluster scope (pairs with mbar_arrive_remote).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void tmap_prefetch(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// Barrier of the 256 consumer threads (the producer warp does not take part).
__device__ __forceinline__ void bar_cons() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4s(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// 16-byte streaming weight load, or zeros without a load when `pred` is false.
__device__ __forceinline__ uint4 ld_weights16_pred(const void* p, bool pred) {
  uint4 r;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %5, 0;\n\tmov.b32 %0, 0;\n\tmov.b32 %1, 0;\n\tmov.b32 %2, 0;\n\t"
      "mov.b32 %3, 0;\n\t@q ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "r"(static_cast<int>(pred)));
  return r;
}

// v = t0 + t1 + t2 in the storage type (t0 = rn(v), t1 = rn(v - t0),
// t2 = rn(v - t0 - t1); both differences are exact in fp32): term `which`
// of v.x in the low half, of v.y in the high half.
template <int DT>
__device__ __forceinline__ uint32_t split_term(float2 v, int which) {
  uint32_t out = 0;
#pragma unroll
  for (int s = 0; s < 3; ++s) {
    uint32_t bx, by;
    float rx, ry;
    if constexpr (DT == MOE_BF16) {
      const __nv_bfloat16 hx = __float2bfloat16_rn(v.x), hy = __float2bfloat16_rn(v.y);
      bx = __bfloat16_as_ushort(hx); by = __bfloat16_as_ushort(hy);
      rx = __bfloat162float(hx); ry = __bfloat162float(hy);
    } else {
      const __half hx = __float2half_rn(v.x), hy = __float2half_rn(v.y);
      bx = __half_as_ushort(hx); by = __half_as_ushort(hy);
      rx = __half2float(hx); ry = __half2float(hy);
    }
    if (s == which) out = bx | (by << 16);
    v.x -= rx;
    v.y -= ry;
  }
  return out;
}

template <int DT, int MINB>
__global__ void __launch_bounds__(kStrThreads, MINB)
    decode_stream_kernel(const __grid_constant__ CUtensorMap mapW2, const __grid_constant__ CUtensorMap mapWs2,
                         const StreamArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t s_full[kStrMaxStages];
  __shared__ __align__(8) uint64_t s_empty[kStrMaxStages];
  __shared__ __align__(8) uint64_t s_actbar[kStrMaxUnits];  // partner's 8 activations of a unit are here
  __shared__ __align__(8) uint64_t s_redbar[kStrMaxUnits];  // every warp's W13 partial sums of a unit are in
  __shared__ __align__(8) uint64_t s_ownbar[kStrMaxUnits];  // this CTA's 8 activations of a unit are in act
  __shared__ __align__(8) uint64_t s_routed;                // ids and weights are in s_ids / s_w
  __shared__ int s_ids[8];
  __shared__ float s_sel[8];
  __shared__ float s_w[8];
  __shared__ float s_gate;
  __shared__ uint32_t s_epoch;
  __shared__ volatile uint32_t s_fail;
  __shared__ int s_issued, s_consumed;
  __shared__ unsigned long long s_cand[64];
  __shared__ __align__(16) unsigned long long s_wkey[256];
  __shared__ float s_red[kStrCons][16];         // router partial sums
  __shared__ float s_ured[2][kStrCons][16];     // W13 partial sums of a unit (by unit parity)

  uint8_t* ring = smem;
  uint16_t* xh = reinterpret_cast<uint16_t*>(smem + a.off_x);  // x in its storage type
  float* lg = reinterpret_cast<float*>(smem + a.off_lg);        // the E (+1) logits
  float* act = reinterpret_cast<float*>(smem + a.off_act);      // [kStrMaxUnits][16] activations
  float* red = reinterpret_cast<float*>(smem + a.off_red);      // [C][hn] partials of my output rows

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const uint32_t rank = cluster_ctarank();  // which half of every unit this CTA takes
  const int cl = static_cast<int>(cluster_id_x());
  const int H = a.H, E = a.E, k = a.k, I = a.I, Is = a.Is;
  const int Hh = H >> 1;
  const size_t rowb = static_cast<size_t>(H) * 2;
  const int nu = cl < a.U ? (a.U - 1 - cl) / a.C + 1 : 0;  // units of this cluster: cl + q*C
  const int nst = 3 * nu;                                  // W13 half 0, W13 half 1, W2 per unit
  const int upe = I >> 4;                                  // units per routed expert
  const int NS = a.NS;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kStrCons);
    }
    for (int i = 0; i < kStrMaxUnits; ++i) {
      mbar_init(&s_actbar[i], 1);
      mbar_init(&s_redbar[i], kStrCons);
      mbar_init(&s_ownbar[i], 1);
    }
    mbar_init(&s_routed, 1);
    s_fail = 0;
    s_issued = 0;
    s_consumed = 1 << 30;
    mbar_fence_init();
  }
  MOE_STAMP(0);  // entry
  if (tid < ((H * 2 + 127) >> 7)) prefetch_l2(a.x + 128 * static_cast<size_t>(tid));
  if (tid == kStrThreads - 1) prefetch_l2(&a.ctrl->gen);
  pdl_launch_dependents();
  __syncthreads();
  cluster_arrive();  // this CTA's barriers are initialised (the partner waits for it before arriving on them)

  // ------------------------------------------------------------ producer
  if (warp == kStrCons) {
    tmap_prefetch(&mapW2);
    tmap_prefetch(&mapWs2);
    // unit of stage idx, and its expert and first column
    auto issue = [&](int idx) {
      const int slot = idx % NS, part = idx % 3;
      const int u = cl + (idx / 3) * a.C;
      uint8_t* dst = ring + static_cast<size_t>(slot) * a.stage_bytes;
      const bool shared = u < a.Us;
      const int q = u - a.Us;
      const int j = shared ? 0 : q / upe;
      const int i0 = shared ? 16 * u : 16 * (q - j * upe);
      const int e = shared ? 0 : s_ids[j];
      if (lane == 0) mbar_arrive_expect_tx(&s_full[slot], 16u * static_cast<uint32_t>(H));
      __syncwarp();
      if (part < 2) {
        if (lane < 16) {
          const int iu = shared ? Is : I;
          const int row = (lane < 8 ? 0 : iu) + i0 + 8 * static_cast<int>(rank) + (lane & 7);
          const uint8_t* base = shared ? a.sw13 : a.w13 + static_cast<size_t>(e) * 2 * I * rowb;
          bulk_g2s(dst + lane * a.pitch, base + static_cast<size_t>(row) * rowb + static_cast<size_t>(part) * H,
                   static_cast<uint32_t>(H), &s_full[slot]);
        }
      } else {
        const int nb = Hh / a.box_rows;
        if (lane < nb) {
          const int y = static_cast<int>(rank) * Hh + lane * a.box_rows;
          if (shared) tma_2d(dst + lane * a.box_rows * 32, &mapWs2, &s_full[slot], i0, y);
          else tma_2d(dst + lane * a.box_rows * 32, &mapW2, &s_full[slot], i0, e * H + y);
        }
      }
    };
    int idx = 0;
    // static weights: the leading shared-expert stages go out before the wait
    if (a.static_weights)
      for (; idx < nst && idx < NS && cl + (idx / 3) * a.C < a.Us; ++idx) issue(idx);
    pdl_wait();
    cluster_wait();
    bool routed = false;
    for (; idx < nst; ++idx) {
      if (!routed && cl + (idx / 3) * a.C >= a.Us) {
        const uint64_t dl = global_ns() + a.timeout_ns;
        bool ok = true;
        while (!mbar_try_wait(&s_routed, 0)) {
          if (global_ns() > dl) { ok = false; break; }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok || s_fail) {
          if (lane == 0 && !ok) s_fail = kDevTimeoutLogits;
          break;
        }
        routed = true;
      }
      if (idx >= NS) {
        const uint32_t par = static_cast<uint32_t>((idx / NS) - 1) & 1u;
        const uint64_t dl = global_ns() + a.timeout_ns;
        bool ok = true;
        while (!mbar_try_wait(&s_empty[idx % NS], par)) {
          if (s_fail || global_ns() > dl) { ok = false; break; }
        }
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0 && !s_fail) s_fail = kDevTimeoutCopy;
          break;
        }
      }
      issue(idx);
    }
    if (lane == 0) s_issued = idx;
  } else {
    // ---------------------------------------------------------- consumers
    const int E1 = E + a.has_gate;
    const int nR = cta < E1 ? (E1 - 1 - cta) / G + 1 : 0;  // <= kStrMaxRouterRows (checked on the host)
    const int nch = H >> 3;                                // 16-byte chunks of a row
    uint4 rw[kStrMaxRouterRows][2];
    auto load_router = [&]() {
#pragma unroll
      for (int r = 0; r < kStrMaxRouterRows; ++r)
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int c = tid + 256 * q;
          const int row = min(cta + r * G, E);
          const bool v = r < nR && c < nch;
          const uint8_t* p = row < E ? a.wr + static_cast<size_t>(row) * rowb : a.swg;
          rw[r][q] = ld_weights16_pred(p + 16 * static_cast<size_t>(v ? c : 0), v);
        }
    };
    if (a.static_weights) load_router();
    pdl_wait();
    MOE_STAMP(1);  // PDL wait released
    if (!a.static_weights) load_router();
    uint32_t gen_prev = 0;
    if (tid == 0) gen_prev = ld_relaxed_u32(&a.ctrl->gen);  // in flight together with x
    for (int c = tid; c < nch; c += 256)
      *reinterpret_cast<uint4*>(xh + 8 * c) = ld_ordered16(a.x + 16 * static_cast<size_t>(c));
    if (tid == 0) {
      const uint32_t ep = gen_prev + 1u;
      s_epoch = ep ? ep : 1u;
    }
    bar_cons();
    const uint32_t epoch = s_epoch;
    MOE_STAMP(2);  // x staged

    // ---- router rows of this CTA: u = cta + r*G (row E is the shared gate)
    {
      float d[kStrMaxRouterRows];
#pragma unroll
      for (int r = 0; r < kStrMaxRouterRows; ++r) d[r] = 0.0f;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c = tid + 256 * q;
        if (c < nch) {
          float xf[8];
          unpack8<DT>(*reinterpret_cast<const uint4*>(xh + 8 * c), xf);
#pragma unroll
          for (int r = 0; r < kStrMaxRouterRows; ++r) {
            float wf[8];
            unpack8<DT>(rw[r][q], wf);
#pragma unroll
            for (int e = 0; e < 8; ++e) d[r] = fmaf(wf[e], xf[e], d[r]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kStrMaxRouterRows; ++r) {
        const float v = warp_sum(d[r]);
        if (lane == 0) s_red[warp][r] = v;
      }
      bar_cons();
      if (tid < 8 * nR) {
        const int r = tid >> 3, rep = tid & 7;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kStrCons; ++w) v += s_red[w][r];
        ll_store(a.ll_logits + static_cast<size_t>(rep) * a.ll_stride + cta + r * G, v, epoch);
      }
    }
    MOE_STAMP(3);  // router rows published

    // ---- routing: gather the logits, rank them (unique 64-bit keys: logit
    // key, then ~index, so the lower index wins ties), weights
    if (warp == 0) {
      const uint64_t* src = a.ll_logits + static_cast<size_t>(cta % kLogitReplicas) * a.ll_stride;
      const bool ok = ll_gather<8>(src, lg, E1, lane, 32, epoch, global_ns() + a.timeout_ns);
      if (!__all_sync(0xffffffffu, ok) && lane == 0) s_fail = kDevTimeoutLogits;
      // every CTA read the epoch before publishing its router rows (G <= E + 1,
      // so each published one), so the next launch may take the next epoch
      if (cta == 0 && lane == 0) atomicExch(&a.ctrl->gen, epoch);
      MOE_STAMP(4);  // logits gathered
    }
    bar_cons();
    {
      const int i0 = warp * 32 + lane;
      const float v0 = lg[min(i0, E - 1)];
      const uint32_t key = i0 < E ? order_key(v0) : 0u;
      const uint64_t mk = key ? (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~i0) : 0ull;
      s_wkey[i0] = mk;
      if (lane < 8) s_cand[warp * 8 + lane] = 0ull;
      __syncwarp();
      int rk = 0;
      const ulonglong2* wk = reinterpret_cast<const ulonglong2*>(s_wkey + warp * 32);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const ulonglong2 kk = wk[j];
        rk += (kk.x > mk ? 1 : 0) + (kk.y > mk ? 1 : 0);
      }
      if (mk != 0ull && rk < k) s_cand[warp * 8 + rk] = mk;
      bar_cons();
      const int c = tid >> 2, q4 = tid & 3;
      const uint64_t kc = s_cand[c];
      int cnt = 0;
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) cnt += s_cand[4 * jj + q4] > kc ? 1 : 0;
      cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
      cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
      if (q4 == 0 && kc != 0ull && cnt < k) {
        const int id = rank_key_index(kc);
        s_ids[cnt] = id;
        s_sel[cnt] = lg[id];
      }
    }
    bar_cons();
    MOE_STAMP(5);  // ranked
    if (warp == 0) {
      if (!s_fail) {
        warp_routing_weights(lg, E, s_sel, k, a.norm_topk, s_w);
        if (lane == 0) s_gate = a.has_gate ? sigmoid_f(lg[E]) : 1.0f;
        __syncwarp();
        if (cta == 0 && lane < k) {
          a.topk_ids[lane] = s_ids[lane];
          a.topk_w[lane] = s_w[lane];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_routed);  // the producer may issue routed stages (or stop on failure)
    }
    bar_cons();
    MOE_STAMP(6);  // routing weights ready
    cluster_wait();  // the partner's barriers are initialised

    // ---- the stages: W13 half 0, W13 half 1, W2 of each unit.  Warps meet
    // only on mbarriers with bounded waits (never on a CTA barrier), so a warp
    // that gives up after an error cannot leave the others blocked.
    const int g = lane >> 2, t = lane & 3;
    const int ksw = (Hh >> 4) / kStrCons;  // k-steps of a W13 stage per warp = m-tiles of a W2 stage per warp
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float pacc[kStrMaxMt][2];
#pragma unroll
    for (int m = 0; m < kStrMaxMt; ++m) pacc[m][0] = pacc[m][1] = 0.0f;
    const uint32_t act_a = smem_u32(act);
    // bounded wait on phase `par` of a barrier (warp-uniform result); records
    // `code` when it runs out
    auto wait_bar = [&](uint64_t* bar, uint32_t par, bool cluster_scope, uint32_t code) -> bool {
      const uint64_t dl = global_ns() + a.timeout_ns;
      bool ok = true;
      while (!(cluster_scope ? mbar_try_wait_cluster(bar, par) : mbar_try_wait(bar, par))) {
        if (s_fail || global_ns() > dl) { ok = false; break; }
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok && lane == 0 && !s_fail) s_fail = code;
      return ok;
    };
    int idx = 0;
    for (; idx < nst; ++idx) {
      if (s_fail) break;
      const int slot = idx % NS;
      if (!wait_bar(&s_full[slot], static_cast<uint32_t>(idx / NS) & 1u, false, kDevTimeoutCopy)) break;
      const int part = idx % 3, ul = idx / 3;
      const int u = cl + ul * a.C;
      const uint32_t sb = smem_u32(ring + static_cast<size_t>(slot) * a.stage_bytes);
      if (part < 2) {
        // 16 rows (gate rows 0-7, up rows 8-15) x this warp's k-steps of the half
        const uint32_t arow = sb + static_cast<uint32_t>(lane & 15) * a.pitch + (lane >> 4) * 16;
        const uint16_t* xb = xh + part * Hh + 2 * t;
        for (int ks = 0; ks < ksw; ++ks) {
          const int kk = (warp * ksw + ks) * 16;
          uint32_t a0, a1, a2, a3;
          ldsm_x4s(arow + 2 * kk, a0, a1, a2, a3);
          uint32_t b0 = 0, b1 = 0;
          if (lane < 4) {
            b0 = *reinterpret_cast<const uint32_t*>(xb + kk);
            b1 = *reinterpret_cast<const uint32_t*>(xb + kk + 8);
          }
          mma16816<DT>(acc, a0, a1, a2, a3, b0, b1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[slot]);
        if (part == 1) {
          // this warp's share of the unit's 16 dot products (column 0 of D)
          if (t == 0) {
            s_ured[ul & 1][warp][g] = acc[0];
            s_ured[ul & 1][warp][8 + g] = acc[2];
          }
          acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_redbar[ul]);
          if (warp == 0) {
            // the unit's 8 activations of this CTA: silu(gate) * up * (routing
            // weight, or the shared gate), kept here and written to the partner
            if (!wait_bar(&s_redbar[ul], 0, false, kDevTimeoutAct)) break;
            if (lane < 8) {
              float gs = 0.0f, us = 0.0f;
#pragma unroll
              for (int w = 0; w < kStrCons; ++w) {
                gs += s_ured[ul & 1][w][lane];
                us += s_ured[ul & 1][w][8 + lane];
              }
              const float sc = u < a.Us ? s_gate : s_w[min((u - a.Us) / upe, k - 1)];
              act[ul * 16 + 8 * rank + lane] = silu_f(gs) * us * sc;
            }
            __syncwarp();
            if (lane == 0) {
              const uint32_t other = rank ^ 1u;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint32_t la = act_a + 4u * static_cast<uint32_t>(ul * 16 + 8 * rank + i);
                st_cluster_f32(mapa_shared(la, other), act[ul * 16 + 8 * rank + i]);
              }
              mbar_arrive_remote(mapa_shared(smem_u32(&s_actbar[ul]), other));
              mbar_arrive(&s_ownbar[ul]);  // releases the local activations to the other warps
            }
          }
        }
      } else {
        // the unit's W2 rows of this CTA's half x its 16 activations (this
        // CTA's 8 and the partner's 8)
        if (!wait_bar(&s_ownbar[ul], 0, false, kDevTimeoutAct)) break;
        if (!wait_bar(&s_actbar[ul], 0, true, kDevTimeoutAct)) break;
        const float* au = act + ul * 16;
        float sc = 1.0f, unsc = 1.0f;
        if constexpr (DT == MOE_F16) {
          // fp16 terms: scale by a power of two that puts the unit's largest
          // magnitude in [2^14, 2^15) (exact, undone on the sums)
          float mx = 0.0f;
#pragma unroll
          for (int i = 0; i < 16; ++i) mx = fmaxf(mx, fabsf(au[i]));
          const uint32_t amax = __float_as_uint(mx);
          int sh = amax ? 14 - (static_cast<int>(amax >> 23) - 127) : 0;
          sh = max(-100, min(100, sh));
          sc = __int_as_float((127 + sh) << 23);
          unsc = __int_as_float((127 - sh) << 23);
        }
        uint32_t b0 = 0, b1 = 0;
        if (g < 3) {
          b0 = split_term<DT>(make_float2(au[2 * t] * sc, au[2 * t + 1] * sc), g);
          b1 = split_term<DT>(make_float2(au[2 * t + 8] * sc, au[2 * t + 9] * sc), g);
        }
        const uint32_t arow = sb + static_cast<uint32_t>(lane & 15) * 32 + (lane >> 4) * 16;
#pragma unroll
        for (int m = 0; m < kStrMaxMt; ++m) {
          if (m < ksw) {
            const int m0 = (warp * ksw + m) * 16;
            uint32_t a0, a1, a2, a3;
            ldsm_x4s(arow + 32u * static_cast<uint32_t>(m0), a0, a1, a2, a3);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            mma16816<DT>(d, a0, a1, a2, a3, b0, b1);
            // columns 0-2 (the three terms) of rows g and g + 8: lane t = 0
            // holds columns 0, 1, lane t = 1 column 2 (column 3 is zero)
            float top = t == 0 ? d[0] + d[1] : (t == 1 ? d[0] : 0.0f);
            float bot = t == 0 ? d[2] + d[3] : (t == 1 ? d[2] : 0.0f);
            top += __shfl_xor_sync(0xffffffffu, top, 1);
            bot += __shfl_xor_sync(0xffffffffu, bot, 1);
            pacc[m][0] += top * unsc;
            pacc[m][1] += bot * unsc;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[slot]);
      }
      if (idx == 0) MOE_STAMP(7);  // first stage done
    }
    if (lane == 0) atomicMin(&s_consumed, idx);  // the least any warp got to
    MOE_STAMP(8);  // stages done

    // ---- publish this CTA's partial output rows [rank*H/2, (rank+1)*H/2)
    if (t == 0) {
#pragma unroll
      for (int m = 0; m < kStrMaxMt; ++m) {
        if (m < ksw) {
          const int h = static_cast<int>(rank) * Hh + (warp * ksw + m) * 16 + g;
          ll_store(a.ll_part + static_cast<size_t>(cl) * H + h, pacc[m][0], epoch);
          ll_store(a.ll_part + static_cast<size_t>(cl) * H + h + 8, pacc[m][1], epoch);
        }
      }
    }
    MOE_STAMP(9);  // partials published

    // ---- my output rows [h0, h0 + hn): the sum over the C clusters' partials
    const int h0 = static_cast<int>((static_cast<long long>(H) * cta) / G);
    const int hn = static_cast<int>((static_cast<long long>(H) * (cta + 1)) / G) - h0;
    const int nw = a.C * hn;  // <= 256 * kStrGather (checked on the host)
    {
      const uint64_t dl = global_ns() + a.timeout_ns;
      uint64_t w[kStrGather];
      uint32_t want = 0;
#pragma unroll
      for (int r = 0; r < kStrGather; ++r) {
        const int q = tid + 256 * r;
        const bool in = q < nw;
        const int c = in ? q / hn : 0;
        const int i = in ? q - c * hn : 0;
        want |= (in ? 1u : 0u) << r;
        w[r] = ll_load1_pred(a.ll_part + static_cast<size_t>(c) * H + h0 + i, in);
      }
      bool ok = true;
      for (;;) {
        uint32_t missing = 0;
#pragma unroll
        for (int r = 0; r < kStrGather; ++r) {
          const bool wanted = (want >> r) & 1u;
          const bool good = wanted && static_cast<uint32_t>(w[r] >> 32) == epoch;
          if (good) red[tid + 256 * r] = __uint_as_float(static_cast<uint32_t>(w[r]));
          missing |= (wanted && !good ? 1u : 0u) << r;
        }
        want = missing;
        if (!__any_sync(0xffffffffu, want != 0u)) break;
        if (__any_sync(0xffffffffu, s_fail != 0 || global_ns() > dl)) { ok = false; break; }
#pragma unroll
        for (int r = 0; r < kStrGather; ++r) {
          const int q = tid + 256 * r;
          const bool re = (want >> r) & 1u;
          const int c = re ? q / hn : 0;
          const int i = re ? q - c * hn : 0;
          w[r] = ll_load1_pred(a.ll_part + static_cast<size_t>(c) * H + h0 + i, re);
        }
      }
      if (!ok && lane == 0 && !s_fail) s_fail = kDevTimeoutAct;
    }
    bar_cons();
    MOE_STAMP(10);  // partials gathered
    if (!s_fail && tid < hn) {
      float sum = 0.0f;
      for (int c = 0; c < a.C; ++c) sum += red[c * hn + tid];
      if (a.residual) {
        const uint16_t xb = xh[h0 + tid];
        sum += DT == MOE_BF16 ? __uint_as_float(static_cast<uint32_t>(xb) << 16)
                              : __half2float(__ushort_as_half(xb));
      }
      store_out(a.out, h0 + tid, sum, a.out_dtype);
    }
    MOE_STAMP(11);  // output written
  }

  // ---- teardown: no copy may still be landing, and the partner must be done
  // writing into this CTA's shared memory, before the CTA exits
  __syncthreads();
  if (tid == 0) {
    const uint64_t dl = global_ns() + a.timeout_ns;
    for (int idx = s_consumed; idx < s_issued; ++idx) {
      const uint32_t par = static_cast<uint32_t>(idx / NS) & 1u;
      while (!mbar_try_wait(&s_full[idx % NS], par)) {
        if (global_ns() > dl) {
          if (!s_fail) s_fail = kDevTimeoutCopy;
          break;
        }
      }
    }
    if (s_fail) report_error(a.ctrl, s_fail, static_cast<uint32_t>(cta));
  }
  __syncthreads();
  cluster_arrive();
  cluster_wait();
}

// ------------------------------------------------------------------ host side
namespace {

struct StreamPlan {
  int C = 0, U = 0, Us = 0, G = 0, NS = 0, nu_max = 0, hn_max = 0, box_rows = 0;
  uint32_t pitch = 0, stage_bytes = 0, off_x = 0, off_lg = 0, off_act = 0, off_red = 0;
  size_t smem = 0;
  bool two_per_sm = false;
};

bool stream_shape_ok(const moe_cfg_t& c) {
  const int E1 = c.n_experts + c.has_shared_gate;
  return (c.dtype == MOE_F16 || c.dtype == MOE_BF16) && c.hidden % 256 == 0 && c.hidden <= 4096 &&
         c.inter % 16 == 0 && c.shared_inter % 16 == 0 && c.n_experts <= 256 && c.top_k <= 8 && E1 >= 2;
}

bool make_plan(const moe_cfg_t& c, StreamPlan& p) {
  if (!stream_shape_ok(c)) return false;
  const int H = c.hidden, E1 = c.n_experts + c.has_shared_gate;
  p.Us = c.shared_inter / 16;
  p.U = (c.top_k * c.inter) / 16 + p.Us;
  int C = sm_count() / 2;
  if (C > p.U) C = p.U;
  if (C > kStreamMaxClusters) C = kStreamMaxClusters;
  if (2 * C > E1) C = E1 / 2;  // every CTA computes at least one router row
  if (C < 1) return false;
  p.C = C;
  p.G = 2 * C;
  p.nu_max = (p.U + C - 1) / C;
  if (p.nu_max > kStrMaxUnits) return false;
  if ((E1 + p.G - 1) / p.G > kStrMaxRouterRows) return false;
  p.hn_max = (H + p.G - 1) / p.G;
  if (p.C * p.hn_max > 256 * kStrGather) return false;
  p.box_rows = H / 2 < 256 ? H / 2 : 256;
  p.pitch = static_cast<uint32_t>(H + 16);
  p.stage_bytes = static_cast<uint32_t>(align_up(16 * static_cast<size_t>(p.pitch), 128));
  const int nst = 3 * p.nu_max;
  // a ring small enough for two CTAs per SM when the CTA's whole stage list
  // fits in three stages (the next layer's CTA then sits beside this one and
  // starts its routing-independent copies early); else the deepest ring
  for (int pass = 0; pass < 2; ++pass) {
    p.NS = pass == 0 ? (nst < 3 ? nst : 3) : (nst < kStrMaxStages ? nst : kStrMaxStages);
    size_t off = static_cast<size_t>(p.NS) * p.stage_bytes;
    p.off_x = static_cast<uint32_t>(off);
    off += align_up(static_cast<size_t>(H) * 2, 128);
    p.off_lg = static_cast<uint32_t>(off);
    off += align_up((c.n_experts + 2) * 4, 128);
    p.off_act = static_cast<uint32_t>(off);
    off += kStrMaxUnits * 16 * 4;
    p.off_red = static_cast<uint32_t>(off);
    off += align_up(static_cast<size_t>(p.C) * p.hn_max * 4, 128);
    p.smem = off;
    // two CTAs of 288 threads with about 4 KB of static shared memory each
    p.two_per_sm = pass == 0 && nst <= 3 && p.smem <= 108 * 1024;
    if (p.two_per_sm) return true;
  }
  return p.smem <= 220 * 1024;
}

template <typename K>
int stream_resident_clusters(K kernel, const StreamPlan& p) {
  struct Entry {
    int dev;
    const void* fn;
    size_t smem;
    int C;
    int n;
  };
  static Entry cache[16];
  static int used = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(attr_mutex());
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].fn == reinterpret_cast<const void*>(kernel) && cache[i].smem == p.smem &&
        cache[i].C == p.C)
      return cache[i].n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kStrThreads);
  cfg.dynamicSmemBytes = p.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (used < 16) cache[used++] = Entry{dev, reinterpret_cast<const void*>(kernel), p.smem, p.C, n};
  return n;
}

template <int DT, int MINB>
moe_status_t launch_stream_dt(const StreamArgs& args, const StreamPlan& p, const CUtensorMap& m2,
                              const CUtensorMap& ms2, cudaStream_t st) {
  auto kernel = decode_stream_kernel<DT, MINB>;
  if (raise_smem_limit(kernel, p.smem) != cudaSuccess) return check_launch("cudaFuncSetAttribute(decode_stream)");
  // the pairs wait on one another and every CTA waits for every cluster's
  // partial output, so all of them must be resident at once
  const int fit = stream_resident_clusters(kernel, p);
  if (fit < 0) return set_error(MOE_ERR_CUDA, "decode: cluster occupancy query failed");
  if (fit < p.C)
    return set_error(MOE_ERR_UNSUPPORTED, "decode: %d CTA pairs must be co-resident, the device holds %d", p.C, fit);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kStrThreads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, kernel, m2, ms2, args) != cudaSuccess) return check_launch("decode_stream_kernel");
  stat_kernels(1);
  return MOE_OK;
}

}  // namespace

bool decode_stream_ok(const moe_cfg_t& c) {
  StreamPlan p;
  return tma_encoder_available() && make_plan(c, p);
}

int decode_stream_clusters(const moe_cfg_t& c) {
  StreamPlan p;
  return make_plan(c, p) ? p.C : 0;
}

moe_status_t launch_decode_stream(const moe_cfg_t& c, const BlockPtrs& bp, uint8_t* ws, const WsLayout& L,
                                  cudaStream_t st) {
  StreamPlan p;
  if (!make_plan(c, p)) return set_error(MOE_ERR_UNSUPPORTED, "decode: shape not taken by the streaming kernel");
  const int H = c.hidden, E = c.n_experts, I = c.inter, Is = c.shared_inter;
  CUtensorMap m2, ms2;
  if (!encode_map_2d(&m2, c.dtype, bp.w2, static_cast<uint64_t>(I), static_cast<uint64_t>(E) * H,
                     static_cast<uint64_t>(I) * 2, 16, static_cast<uint32_t>(p.box_rows)))
    return set_error(MOE_ERR_CUDA, "decode: cuTensorMapEncodeTiled failed (W2)");
  if (Is > 0) {
    if (!encode_map_2d(&ms2, c.dtype, bp.shared_w2, static_cast<uint64_t>(Is), static_cast<uint64_t>(H),
                       static_cast<uint64_t>(Is) * 2, 16, static_cast<uint32_t>(p.box_rows)))
      return set_error(MOE_ERR_CUDA, "decode: cuTensorMapEncodeTiled failed (shared W2)");
  } else {
    ms2 = m2;
  }
  StreamArgs a;
  a.x = static_cast<const uint8_t*>(bp.x);
  a.wr = static_cast<const uint8_t*>(bp.router_w);
  a.w13 = static_cast<const uint8_t*>(bp.w13);
  a.sw13 = static_cast<const uint8_t*>(bp.shared_w13);
  a.swg = static_cast<const uint8_t*>(bp.shared_gate_w);
  a.topk_ids = bp.topk_ids;
  a.topk_w = bp.topk_w;
  a.out = bp.out;
  a.ctrl = reinterpret_cast<Control*>(ws + L.ctrl);
  a.ll_logits = reinterpret_cast<uint64_t*>(ws + L.ll_logits);
  a.ll_part = reinterpret_cast<uint64_t*>(ws + L.ll_part);
  a.H = H; a.E = E; a.k = c.top_k; a.I = I; a.Is = Is;
  a.has_gate = c.has_shared_gate; a.norm_topk = c.norm_topk; a.out_dtype = c.out_dtype;
  a.static_weights = (c.flags & MOE_FLAG_STATIC_WEIGHTS) ? 1 : 0;
  a.residual = (c.flags & MOE_FLAG_RESIDUAL) ? 1 : 0;
  a.ll_stride = (E + 2) & ~1;
  a.C = p.C; a.U = p.U; a.Us = p.Us; a.NS = p.NS; a.box_rows = p.box_rows;
  a.pitch = p.pitch; a.stage_bytes = p.stage_bytes;
  a.off_x = p.off_x; a.off_lg = p.off_lg; a.off_act = p.off_act; a.off_red = p.off_red;
  a.timeout_ns = wait_timeout_ns();
#ifdef MOE_PHASE_TRACE
  a.trace = trace_next_record();
  if (!a.trace) return check_launch("trace buffer");
#endif
  if (c.dtype == MOE_BF16)
    return p.two_per_sm ? launch_stream_dt<MOE_BF16, 2>(a, p, m2, ms2, st) : launch_stream_dt<MOE_BF16, 1>(a, p, m2, ms2, st);
  return p.two_per_sm ? launch_stream_dt<MOE_F16, 2>(a, p, m2, ms2, st) : launch_stream_dt<MOE_F16, 1>(a, p, m2, ms2, st);
}

}  // namespace moe
