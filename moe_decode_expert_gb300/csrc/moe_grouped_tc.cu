// moe_grouped_tc.cu — tensor-core (tcgen05 / TMEM / TMA) grouped expert GEMMs
// for T > 1 tokens.
//
// "Decode throughput analysis report", code-level profiling section: the
// prefill routed-expert path is the largest time-to-first-token cost and the
// next step named there is a grouped GEMM over experts; "BI-V100 inference
// work log", Part 7: once the tokens per expert grow, the MoE GEMM becomes a
// real matrix product.  Swap-AB formulation per expert e with m_e tokens:
//
//   W13 pass   D[128 rows, N tokens] = [Wg rows i0..i0+63 ; Wu rows i0..i0+63] . Xs^T
//              (K = H; Xs = x rows in expert order, or x itself for T <= 16),
//              epilogue act = silu(gate) * up for the 64 rows, stored as
//              a two-term split act = hi + lo in the storage dtype (hi = rn(act),
//              lo = rn(act - hi): 16 significant bits) so the next pass keeps
//              fp32-level accuracy of the activation;
//   W2 pass    D[128 rows (h), N tokens] = W2[e][h0..h0+127, :] . (hi + lo)^T
//              (K = I, two MMAs per K step), epilogue y[pair, h] = weight(pair) * D.
//
// Both operands are K-major; tiles are moved by TMA (cp.async.bulk.tensor,
// 128-byte swizzle) into a multi-stage shared-memory ring, multiplied by
// tcgen05.mma (cta_group::1, kind::f16, fp32 accumulators in TMEM, double
// buffered so the epilogue of one tile overlaps the MMAs of the next), and
// read back with tcgen05.ld.  Warp roles: warp 0 issues TMA, warp 1 owns TMEM
// and issues MMAs, warps 2-5 run the epilogue (one TMEM lane quarter each).
// Every mbarrier wait is bounded by the GPU global timer; on expiry the kernel
// records MOE_ERR_TIMEOUT, lets its own copies and MMAs finish (bounded),
// frees its TMEM and returns.

#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_common.cuh"
#include "moe_internal.h"
#include "moe_stages.cuh"

namespace moe {

constexpr int kTcThreads = 192;
constexpr int kBK = 64;                 // K elements per stage: one 128-byte swizzle row
constexpr uint32_t kTileA = 128 * 128;  // 128 rows x 128 bytes
constexpr int kSmemBudget = 220 * 1024;
// Ranked grouping: up to this many pairs the filing launch also copies the x
// rows (T = 64 / 512: 1.0 / 2.6 us less per layer); beyond, a gather launch
// with twice the warps per SM copies them faster (T = 4096: 2.7 us).
constexpr int kFoldGatherMaxPairs = 16384;


// ----------------------------------------------------------------- PTX
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}
// Fetch a tensor map (a __grid_constant__ kernel parameter) ahead of its first
// TMA copy.
__device__ __forceinline__ void tensormap_prefetch(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 lanes x 16 consecutive fp32 columns of TMEM -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// The same load without its wait: a load goes out while earlier values are
// used; tmem_ld_wait() then tmem_ld_tie() on the destination before its first
// use (the tie keeps the compiler from reading the registers above the wait).
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld_tie(uint32_t (&r)[16]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]));
}
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO),
// descriptor version 1, layout "128B swizzle".
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both DT
// (fp16 = 0, bf16 = 1), both K-major, M = 128, N.
template <int DT, int N>
__device__ __forceinline__ constexpr uint32_t idesc_f16() {
  constexpr uint32_t fmt = DT == MOE_BF16 ? 1u : 0u;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(128 >> 4) << 24);
}

template <int DT>
__device__ __forceinline__ void split_store(uint16_t* hi, uint16_t* lo, size_t off, float a) {
  if constexpr (DT == MOE_BF16) {
    const __nv_bfloat16 h = __float2bfloat16_rn(a);
    const __nv_bfloat16 l = __float2bfloat16_rn(a - __bfloat162float(h));
    hi[off] = __bfloat16_as_ushort(h);
    lo[off] = __bfloat16_as_ushort(l);
  } else {
    const __half h = __float2half_rn(a);
    const __half l = __float2half_rn(a - __half2float(h));
    hi[off] = __half_as_ushort(h);
    lo[off] = __half_as_ushort(l);
  }
}

// Bounded wait used by every role; false on timeout or when another role aborted.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, uint64_t timeout, volatile int* abort) {
  const uint64_t deadline = global_ns() + timeout;
  while (!mbar_try_wait(bar, parity)) {
    if (*abort || global_ns() > deadline) return false;
  }
  return true;
}

// OR of `v` over the 128 epilogue threads (named barrier 1 with reduction):
// every epilogue thread gets the same answer, so they leave loops together
// and none is left waiting at a named barrier.
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 128, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// ======================================================= W13 + SiLU pass
// MT 128-row M-tiles (each 64 gate rows stacked on the matching 64 up rows) of
// one expert share every token (B) stage, so the token operand is read from L2
// once per MT M-tiles; each tile has its own TMEM accumulator (2*MT*N columns
// with double buffering).  The token operand is the gathered rows Xs (rows
// pos0.. of the tile's pairs), or with DIRECT (T <= 16) x itself: every tile
// then computes all T token columns and pair j of the tile takes the column of
// its token.  Tiles are taken dynamically as in the W2 pass below.
template <int DT, int N, int MT, bool DIRECT>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_w13_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapAs,
                  const __grid_constant__ CUtensorMap mapB, const TcTile* tiles,
                  const int32_t* n_tiles_p, int H, int I, int Is, int E, int act_stride,
                  uint16_t* __restrict__ act_hi, uint16_t* __restrict__ act_lo, Control* ctrl, uint64_t timeout,
                  const int32_t* perm, int direct_T, int k, int32_t* tile_ctr, int32_t* zero_cnt, int zero_n) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  constexpr uint32_t kStage = MT * kTileA + N * 128;
  constexpr int kStg = 128 * 17 * 4;
  constexpr int kStages = (kSmemBudget - kStg) / kStage > 8 ? 8 : (kSmemBudget - kStg) / kStage;
  constexpr uint32_t kCols = 2 * MT * N;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stg = reinterpret_cast<float*>(smem + kStages * kStage);  // [128][17] epilogue staging
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], done, tq_full[4], tq_empty[4];
  __shared__ int s_tq[4];  // tile queue: the producer's tiles, in order, for the MMA and epilogue warps
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;
  __shared__ int s_tok[DIRECT ? N : 1];  // DIRECT: token of each pair of the current tile

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], 4); }
    for (int a = 0; a < 4; ++a) { mbar_init(&tq_full[a], 1); mbar_init(&tq_empty[a], 2); }
    mbar_init(&done, 1);
    mbar_fence_init();
    s_abort = 0;
    tensormap_prefetch(&mapA);
    tensormap_prefetch(&mapAs);
    tensormap_prefetch(&mapB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The set-up above reads nothing an earlier kernel writes; from here on the
  // tile list and the operands it wrote are read.
  pdl_wait();
  const uint32_t tbase = tmem_base_s;
  const int ntiles = *n_tiles_p;
  const int KB = H / kBK;
  // the ranked grouping's per-expert counters, read by the filing launch before
  // this one, start the next call at zero
  if (zero_cnt && blockIdx.x == 0)
    for (int e = threadIdx.x; e < zero_n; e += kTcThreads) zero_cnt[e] = 0;

  if (warp == 0) {
    if (lane == 0) {  // ---------------------------------------------- TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      for (int j = 0; !s_abort; ++j) {
        const int qs = j & 3;
        if (j >= 4 && !tc_wait(&tq_empty[qs], ((j >> 2) - 1) & 1, timeout, &s_abort)) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        int t = j == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(tile_ctr, 1);
        if (t >= ntiles) t = -1;
        s_tq[qs] = t;
        mbar_arrive(&tq_full[qs]);
        if (t < 0) break;
        const TcTile tl = tiles[t];
        const bool sh = tl.e == E;
        const CUtensorMap* mA = sh ? &mapAs : &mapA;
        const int ie = sh ? Is : I;
        const int m0 = tl.m * MT;
        const int nv = min(MT, ie / 64 - m0);
        const int rowg = (sh ? 0 : tl.e * 2 * I) + m0 * 64;
        const uint32_t bytes = static_cast<uint32_t>(nv) * kTileA + N * 128;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc_wait(&empty[stage], phase ^ 1u, timeout, &s_abort)) {
            s_abort = 1;
            report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
            break;
          }
          uint8_t* sA = smem + stage * kStage;
          mbar_arrive_expect_tx(&full[stage], bytes);
          for (int mt = 0; mt < nv; ++mt) {
            tma_load_2d(sA + mt * kTileA, mA, &full[stage], kb * kBK, rowg + mt * 64);
            tma_load_2d(sA + mt * kTileA + kTileA / 2, mA, &full[stage], kb * kBK, rowg + mt * 64 + ie);
          }
          tma_load_2d(sA + MT * kTileA, &mapB, &full[stage], kb * kBK, DIRECT ? 0 : tl.pos0);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // let every copy this thread issued land before the CTA exits
      for (int s = 0; s < kStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait_until(&full[s], (issued_phase >> s) & 1u, global_ns() + timeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_f16<DT, N>();
      int stage = 0;
      uint32_t phase = 0;
      for (int it = 0; !s_abort; ++it) {
        const int qs = it & 3;
        if (!tc_wait(&tq_full[qs], (it >> 2) & 1, timeout, &s_abort)) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        const int t = s_tq[qs];
        mbar_arrive(&tq_empty[qs]);
        if (t < 0) break;
        const TcTile tl = tiles[t];
        const int ie = tl.e == E ? Is : I;
        const int nv = min(MT, ie / 64 - tl.m * MT);
        const int acc = it & 1;
        if (!tc_wait(&tempty[acc], ((it >> 1) & 1) ^ 1u, timeout, &s_abort)) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc_wait(&full[stage], phase, timeout, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * kStage);
          const uint32_t sB = sA + MT * kTileA;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
              if (mt < nv)
                tc_mma(tbase + static_cast<uint32_t>((acc * MT + mt) * N), sw128_desc(sA + mt * kTileA + 32 * k),
                       sw128_desc(sB + 32 * k), idesc, (kb | k) != 0);
          tc_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        tc_commit(&tfull[acc]);
      }
      tc_commit(&done);  // completes once every MMA issued above has completed
      mbar_wait_until(&done, 0, global_ns() + timeout);
    }
  } else {  // ---------------------------------------------------- epilogue, 128 threads
    const int q = warp & 3;
    const int row = 32 * q + lane;          // TMEM lane this thread reads
    const int etid = threadIdx.x - 64;      // 0..127
    const int ar = etid & 63, half = etid >> 6;  // activation row and column half it computes
    for (int it = 0;; ++it) {
      const int qs = it & 3;
      const bool okq = !s_abort && tc_wait(&tq_full[qs], (it >> 2) & 1, timeout, &s_abort);
      const int t = okq ? s_tq[qs] : -1;
      if (epi_any(!okq)) {  // every epilogue thread has read the queue entry
        s_abort = 1;
        report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
        break;
      }
      if (etid == 0) mbar_arrive(&tq_empty[qs]);
      if (t < 0) break;
      const TcTile tl = tiles[t];
      const int ie = tl.e == E ? Is : I;
      const int nv = min(MT, ie / 64 - tl.m * MT);
      const int acc = it & 1;
      if constexpr (DIRECT)  // token (accumulator column) of each pair of the tile
        for (int c = etid; c < tl.n; c += 128) {
          const int p = perm[tl.pos0 + c];
          s_tok[c] = p < direct_T * k ? p / k : p - direct_T * k;
        }
      const bool ok = !s_abort && tc_wait(&tfull[acc], (it >> 1) & 1, timeout, &s_abort);
      if (epi_any(!ok)) {
        s_abort = 1;
        report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
        break;
      }
      tc_fence_after();
      for (int mt = 0; mt < nv; ++mt) {
        const int i = (tl.m * MT + mt) * 64 + ar;
        const int ncols = DIRECT ? direct_T : tl.n;  // accumulator columns holding results
        const uint32_t ta = tbase + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>((acc * MT + mt) * N);
        // 16 columns at a time through the staging rows; the next block's TMEM
        // load is in flight meanwhile (two register blocks in turn)
        auto block = [&](const uint32_t (&v)[16], int c0) {
#pragma unroll
          for (int j = 0; j < 16; ++j) stg[row * 17 + j] = __uint_as_float(v[j]);
          named_bar_sync(1, 128);
          if constexpr (DIRECT) {
            // column = token: pair j of the tile takes its token's column
            for (int j = half; j < tl.n; j += 2) {
              const int col = s_tok[j] - c0;
              if (col >= 0 && col < 16) {
                const float g = stg[ar * 17 + col], u = stg[(ar + 64) * 17 + col];
                split_store<DT>(act_hi, act_lo, static_cast<size_t>(tl.pos0 + j) * act_stride + i, silu_f(g) * u);
              }
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int j = half * 8 + jj;
              const int col = c0 + j;
              if (col < tl.n) {
                const float g = stg[ar * 17 + j], u = stg[(ar + 64) * 17 + j];
                split_store<DT>(act_hi, act_lo, static_cast<size_t>(tl.pos0 + col) * act_stride + i, silu_f(g) * u);
              }
            }
          }
          named_bar_sync(1, 128);
        };
        uint32_t va[16], vb[16];
        tmem_ld16_issue(ta, va);
        tmem_ld_wait();
        tmem_ld_tie(va);
        for (int c0 = 0; c0 < ncols; c0 += 32) {
          if (c0 + 16 < ncols) tmem_ld16_issue(ta + c0 + 16, vb);
          block(va, c0);
          tmem_ld_wait();
          tmem_ld_tie(vb);
          if (c0 + 16 < ncols) {
            if (c0 + 32 < ncols) tmem_ld16_issue(ta + c0 + 32, va);
            block(vb, c0 + 16);
            tmem_ld_wait();
            tmem_ld_tie(va);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kCols);
  }
}

// =========================================================== W2 pass
// MT 128-row M-tiles of W2 (output rows h) of one expert share every
// activation (hi, lo) stage.  Tiles are taken dynamically: CTA c starts with
// tile c, then the producer takes the next from a global counter (SMs that
// finish early take more) and passes each tile to the MMA and epilogue warps
// through a 4-entry shared-memory queue (tq_full / tq_empty).
template <int DT, int N, int MT>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_w2_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapAs,
                 const __grid_constant__ CUtensorMap mapHi, const __grid_constant__ CUtensorMap mapLo,
                 const __grid_constant__ CUtensorMap mapHiS, const __grid_constant__ CUtensorMap mapLoS,
                 const TcTile* tiles, const int32_t* n_tiles_p,
                 const int32_t* perm, const float* topk_w,
                 const float* gate_logits, int gate_stride, int has_gate, int T, int H, int I, int Is,
                 int E, int k, float* __restrict__ y, int32_t* tile_ctr, Control* ctrl, uint64_t timeout) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  constexpr uint32_t kStage = MT * kTileA + 2 * N * 128;
  constexpr int kStages = kSmemBudget / kStage > 8 ? 8 : kSmemBudget / kStage;
  constexpr uint32_t kCols = 2 * MT * N;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], done, tq_full[4], tq_empty[4];
  __shared__ int s_tq[4];
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;
  __shared__ int s_pair[N];
  __shared__ float s_wt[N];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], 4); }
    for (int a = 0; a < 4; ++a) { mbar_init(&tq_full[a], 1); mbar_init(&tq_empty[a], 2); }
    mbar_init(&done, 1);
    mbar_fence_init();
    s_abort = 0;
    tensormap_prefetch(&mapA);
    tensormap_prefetch(&mapAs);
    tensormap_prefetch(&mapHi);
    tensormap_prefetch(&mapLo);
    tensormap_prefetch(&mapHiS);
    tensormap_prefetch(&mapLoS);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The set-up above reads nothing an earlier kernel writes; from here on the
  // tile list and the operands it wrote are read.
  pdl_wait();
  const uint32_t tbase = tmem_base_s;
  const int ntiles = *n_tiles_p;
  const int mtiles = H / 128;

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      for (int j = 0; !s_abort; ++j) {
        const int qs = j & 3;
        if (j >= 4 && !tc_wait(&tq_empty[qs], ((j >> 2) - 1) & 1, timeout, &s_abort)) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        int t = j == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(tile_ctr, 1);
        if (t >= ntiles) t = -1;
        s_tq[qs] = t;
        mbar_arrive(&tq_full[qs]);
        if (t < 0) break;
        const TcTile tl = tiles[t];
        const bool sh = tl.e == E;
        const CUtensorMap* mA = sh ? &mapAs : &mapA;
        const CUtensorMap* mH = sh ? &mapHiS : &mapHi;
        const CUtensorMap* mL = sh ? &mapLoS : &mapLo;
        const int KB = (sh ? Is : I) / kBK;
        const int m0 = tl.m * MT;
        const int nv = min(MT, mtiles - m0);
        const int rowa = (sh ? 0 : tl.e * H) + m0 * 128;
        const uint32_t bytes = static_cast<uint32_t>(nv) * kTileA + 2 * N * 128;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc_wait(&empty[stage], phase ^ 1u, timeout, &s_abort)) {
            s_abort = 1;
            report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
            break;
          }
          uint8_t* sA = smem + stage * kStage;
          mbar_arrive_expect_tx(&full[stage], bytes);
          for (int mt = 0; mt < nv; ++mt) tma_load_2d(sA + mt * kTileA, mA, &full[stage], kb * kBK, rowa + mt * 128);
          tma_load_2d(sA + MT * kTileA, mH, &full[stage], kb * kBK, tl.pos0);
          tma_load_2d(sA + MT * kTileA + N * 128, mL, &full[stage], kb * kBK, tl.pos0);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < kStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait_until(&full[s], (issued_phase >> s) & 1u, global_ns() + timeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16<DT, N>();
      int stage = 0;
      uint32_t phase = 0;
      for (int it = 0; !s_abort; ++it) {
        const int qs = it & 3;
        if (!tc_wait(&tq_full[qs], (it >> 2) & 1, timeout, &s_abort)) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        const int t = s_tq[qs];
        mbar_arrive(&tq_empty[qs]);
        if (t < 0) break;
        const TcTile tl = tiles[t];
        const int KB = (tl.e == E ? Is : I) / kBK;
        const int nv = min(MT, mtiles - tl.m * MT);
        const int acc = it & 1;
        if (!tc_wait(&tempty[acc], ((it >> 1) & 1) ^ 1u, timeout, &s_abort)) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc_wait(&full[stage], phase, timeout, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * kStage);
          const uint32_t sH = sA + MT * kTileA, sL = sH + N * 128;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
              if (mt < nv) {
                const uint32_t d = tbase + static_cast<uint32_t>((acc * MT + mt) * N);
                tc_mma(d, sw128_desc(sA + mt * kTileA + 32 * kk), sw128_desc(sH + 32 * kk), idesc, (kb | kk) != 0);
                tc_mma(d, sw128_desc(sA + mt * kTileA + 32 * kk), sw128_desc(sL + 32 * kk), idesc, 1u);
              }
          tc_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        tc_commit(&tfull[acc]);
      }
      tc_commit(&done);
      mbar_wait_until(&done, 0, global_ns() + timeout);
    }
  } else {
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const int etid = threadIdx.x - 64;  // 0..127
    for (int it = 0;; ++it) {
      const int qs = it & 3;
      const bool okq = !s_abort && tc_wait(&tq_full[qs], (it >> 2) & 1, timeout, &s_abort);
      const int t = okq ? s_tq[qs] : -1;
      // every epilogue thread has read the queue entry (and the previous
      // tile's readers of s_pair / s_wt are done)
      if (epi_any(!okq)) {
        s_abort = 1;
        report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
        break;
      }
      if (etid == 0) mbar_arrive(&tq_empty[qs]);
      if (t < 0) break;
      const TcTile tl = tiles[t];
      const int nv = min(MT, mtiles - tl.m * MT);
      const int acc = it & 1;
      for (int c = etid; c < tl.n; c += 128) {
        const int p = perm[tl.pos0 + c];
        s_pair[c] = p;
        float wt;
        if (p < T * k) wt = topk_w[p];
        else wt = has_gate ? sigmoid_f(gate_logits[static_cast<size_t>(p - T * k) * gate_stride + E]) : 1.0f;
        s_wt[c] = wt;
      }
      const bool ok = !s_abort && tc_wait(&tfull[acc], (it >> 1) & 1, timeout, &s_abort);
      if (epi_any(!ok)) {  // the barrier also publishes s_pair / s_wt
        s_abort = 1;
        report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
        break;
      }
      tc_fence_after();
      // Two 16-column register blocks in turn: the next block's TMEM load is in
      // flight while the current one is stored.
      for (int mt = 0; mt < nv; ++mt) {
        const int h = (tl.m * MT + mt) * 128 + row;
        const uint32_t ta = tbase + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>((acc * MT + mt) * N);
        uint32_t va[16], vb[16];
        tmem_ld16_issue(ta, va);
        tmem_ld_wait();
        tmem_ld_tie(va);
        for (int c0 = 0; c0 < tl.n; c0 += 32) {
          if (c0 + 16 < tl.n) tmem_ld16_issue(ta + c0 + 16, vb);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < tl.n) y[static_cast<size_t>(s_pair[c0 + j]) * H + h] = s_wt[c0 + j] * __uint_as_float(va[j]);
          tmem_ld_wait();
          tmem_ld_tie(vb);
          if (c0 + 32 < tl.n) tmem_ld16_issue(ta + c0 + 32, va);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + 16 + j < tl.n)
              y[static_cast<size_t>(s_pair[c0 + 16 + j]) * H + h] = s_wt[c0 + 16 + j] * __uint_as_float(vb[j]);
          tmem_ld_wait();
          tmem_ld_tie(va);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kCols);
  }
}

// ======================================================== router GEMM (large T)
// logits[t, e] = x[t] . Wr[e] for T tokens on tcgen05: router rows are M (128
// per tile), tokens N (128), K = H.  M-tiles [0, mE) cover the E router rows;
// with a shared gate one more M-tile reads the gate vector as a one-row tensor
// (TMA fills the other 127 rows with zeros).  K is split S ways when the
// tiles would leave SMs idle: split s adds K blocks [s KB/S, (s+1) KB/S) and,
// with S > 1, writes its partial sums to part + s T E1 (the top-k kernel adds
// the S partials in split order).  Tile t: m = t % nm, then s, then n.
template <int DT, int N>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_router_kernel(const __grid_constant__ CUtensorMap mapWr, const __grid_constant__ CUtensorMap mapG,
                     const __grid_constant__ CUtensorMap mapX, int T, int H, int E, int E1, int mE, int nm,
                     int S, float* __restrict__ logits, Control* ctrl, uint64_t timeout) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  constexpr uint32_t kStage = kTileA + N * 128;
  constexpr int kStages = kSmemBudget / kStage > 8 ? 8 : kSmemBudget / kStage;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], done;
  __shared__ uint32_t tmem_base_s;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], 4); }
    mbar_init(&done, 1);
    mbar_fence_init();
    s_abort = 0;
    tensormap_prefetch(&mapWr);
    tensormap_prefetch(&mapG);
    tensormap_prefetch(&mapX);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_s, 2 * N);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The set-up above reads nothing an earlier kernel writes; from here on the
  // tile list and the operands it wrote are read.
  pdl_wait();
  const uint32_t tbase = tmem_base_s;
  const int ntiles = nm * S * ((T + N - 1) / N);
  const int KB = H / kBK / S;  // K blocks per split

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_phase = 0;
      for (int t = blockIdx.x; t < ntiles && !s_abort; t += gridDim.x) {
        const int m = t % nm, sp = (t / nm) % S, n = t / (nm * S);
        const bool gate = m >= mE;
        for (int kb = sp * KB; kb < (sp + 1) * KB; ++kb) {
          if (!tc_wait(&empty[stage], phase ^ 1u, timeout, &s_abort)) {
            s_abort = 1;
            report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
            break;
          }
          uint8_t* sA = smem + stage * kStage;
          mbar_arrive_expect_tx(&full[stage], kStage);
          tma_load_2d(sA, gate ? &mapG : &mapWr, &full[stage], kb * kBK, gate ? 0 : m * 128);
          tma_load_2d(sA + kTileA, &mapX, &full[stage], kb * kBK, n * N);
          issued_mask |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s = 0; s < kStages; ++s)
        if (issued_mask & (1u << s)) mbar_wait_until(&full[s], (issued_phase >> s) & 1u, global_ns() + timeout);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16<DT, N>();
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < ntiles && !s_abort; t += gridDim.x, ++it) {
        const int acc = it & 1;
        if (!tc_wait(&tempty[acc], ((it >> 1) & 1) ^ 1u, timeout, &s_abort)) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        tc_fence_after();
        const uint32_t d = tbase + static_cast<uint32_t>(acc * N);
        bool ok = true;
        for (int kb = 0; kb < KB; ++kb) {
          if (!tc_wait(&full[stage], phase, timeout, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + stage * kStage);
          const uint32_t sB = sA + kTileA;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc_mma(d, sw128_desc(sA + 32 * k), sw128_desc(sB + 32 * k), idesc, (kb | k) != 0);
          tc_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) {
          s_abort = 1;
          report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
          break;
        }
        tc_commit(&tfull[acc]);
      }
      tc_commit(&done);
      mbar_wait_until(&done, 0, global_ns() + timeout);
    }
  } else {
    const int q = warp & 3;
    const int row = 32 * q + lane;
    int it = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
      const int m = t % nm, sp = (t / nm) % S, n = t / (nm * S);
      float* dst = logits + static_cast<size_t>(sp) * T * E1;
      const int acc = it & 1;
      const bool ok = !s_abort && tc_wait(&tfull[acc], (it >> 1) & 1, timeout, &s_abort);
      if (epi_any(!ok)) {
        s_abort = 1;
        report_error(ctrl, kDevTimeoutCopy, blockIdx.x);
        break;
      }
      tc_fence_after();
      const bool gate = m >= mE;
      const int e = gate ? E : m * 128 + row;
      const bool write = gate ? row == 0 : e < E;
      for (int c0 = 0; c0 < N; c0 += 16) {
        if (n * N + c0 >= T) break;
        float v[16];
        tmem_ld16(tbase + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(acc * N + c0), v);
        if (write) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = n * N + c0 + j;
            if (tok < T) dst[static_cast<size_t>(tok) * E1 + e] = v[j];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 2 * N);
  }
}

// ================================================ grouping, schedule + gather
// Layout of `sched`: [0] n13, [1] n2 (tile counts of the two passes), [2] / [3]
// their dynamic tile counters; the TcTile lists sit at their own offsets.

// Grouping from ranks (T > kRouteGroupMaxT): the top-k kernel gave every
// routed pair its rank within its expert and left the totals in cnt.  Every
// CTA scans the totals itself; CTA 0 writes both tile lists, the others file
// the pairs (pair p of expert e at position offsets[e] + rank[p]; the shared
// expert's pair of token t at offsets[E] + t), so the lists are not held up
// by CTA 0's share of the pairs (T = 64 / 512: 0.9 / 2.3 us).  With xs set it
// files a pair per warp and copies the pair's x row to Xs[pos] on the way (no
// gather launch), else a pair per thread.  One launch over many SMs instead of
// a single-CTA counting sort and a schedule launch.
__global__ void __launch_bounds__(1024) tc_fill_kernel(const int32_t* ids, const int32_t* rank, const int32_t* cnt,
                                                       int T, int k, int E, int has_shared, int32_t* perm, int I,
                                                       int Is, int H, int N, int mt13, int mt2, int32_t* n13,
                                                       int32_t* n2, TcTile* t13, TcTile* t2, const uint8_t* x,
                                                       uint8_t* __restrict__ xs, Control* ctrl) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  __shared__ int32_t s_cnt[1026], s_off[1026];
  __shared__ int32_t wsum[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = E + 1;  // experts + the shared expert (n <= 1025: two per thread)
  const int e0 = 2 * tid, e1 = 2 * tid + 1;
  const int c0 = e0 < n ? (e0 < E ? cnt[e0] : (has_shared ? T : 0)) : 0;
  const int c1 = e1 < n ? (e1 < E ? cnt[e1] : (has_shared ? T : 0)) : 0;
  int incl = c0 + c1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    wsum[lane] = v;
  }
  __syncthreads();
  const int before = incl - (c0 + c1) + (warp ? wsum[warp - 1] : 0);
  if (e0 < n) { s_cnt[e0] = c0; s_off[e0] = before; }
  if (e1 < n) { s_cnt[e1] = c1; s_off[e1] = before + c0; }
  __syncthreads();
  if (blockIdx.x == 0) {  // CTA 0 writes the tile lists; the others file the pairs
    schedule_stage(s_cnt, s_off, E, I, Is, H, N, mt13, mt2, n13, n2, t13, t2);
    return;
  }
  const int np = T * k, P = np + (has_shared ? T : 0);
  const int cb = blockIdx.x - 1, ncb = gridDim.x - 1;
  if (!xs) {
    for (int p = cb * 1024 + tid; p < P; p += ncb * 1024) {
      if (p < np) {
        const int e = ids[p];
        if (e >= 0 && e < E) perm[s_off[e] + rank[p]] = p;
        else report_error(ctrl, kDevBadExpert, static_cast<uint32_t>(p));
      } else {
        perm[s_off[E] + (p - np)] = p;
      }
    }
    return;
  }
  const int nch = H >> 3;  // 16-byte chunks per x row
  for (int p = cb * 32 + warp; p < P; p += ncb * 32) {
    int pos = 0;
    if (lane == 0) {
      const int e = p < np ? ids[p] : E;
      if (e >= 0 && e <= E) {
        pos = p < np ? s_off[e] + rank[p] : s_off[E] + (p - np);
        perm[pos] = p;
      } else {
        pos = -1;
        report_error(ctrl, kDevBadExpert, static_cast<uint32_t>(p));
      }
    }
    pos = __shfl_sync(0xffffffffu, pos, 0);
    if (pos < 0) continue;
    const int t = p < np ? p / k : p - np;
    const uint8_t* src = x + static_cast<size_t>(t) * H * 2;
    uint8_t* dst = xs + static_cast<size_t>(pos) * H * 2;
    for (int c0 = lane; c0 < nch; c0 += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + 32 * u < nch) v[u] = ld_nc16(src + 16 * (c0 + 32 * u));
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + 32 * u < nch) *reinterpret_cast<uint4*>(dst + 16 * (c0 + 32 * u)) = v[u];
    }
  }
}

// Small batches (T <= 32, E <= 256): the ranking of every token, the counting
// sort of the pairs by expert and the tile lists of both tensor-core passes in
// one single-CTA launch instead of three (each of those kernels is a few µs of
// mostly fixed latency at this size).  All 1024 threads add the router's split
// partial sums (every load in flight at once), warp t ranks token t, then all
// threads group and schedule; ids, counts and offsets pass between the stages
// in shared memory.
// kWarp: the grouping by one warp and the tile lists by every thread (at most
// kWarpGroupPairs pairs with the shared expert); else the CTA-wide stages.  Two
// instantiations, so each launch carries only its own code.
template <bool kWarp>
__global__ void __launch_bounds__(1024) route_group_kernel(float* logits, const float* part,
                                                           int nsplit, int T, int E, int E1, int k, int norm_topk,
                                                           int32_t* ids, float* w, int has_shared, int32_t* counts,
                                                           int32_t* offsets, int32_t* perm, Control* ctrl, int I,
                                                           int Is, int H, int N, int mt13, int mt2, int32_t* n13,
                                                           int32_t* n2, TcTile* t13, TcTile* t2) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  // T <= kRouteGroupMaxT, E1 <= 257, k <= 32 (checked on the host)
  extern __shared__ float s_lg[];  // the T rows of logits [T, E1] (dynamic)
  __shared__ int s_ids[kRouteGroupMaxT][32];
  __shared__ float s_sel[kRouteGroupMaxT][32];
  __shared__ float s_w[kRouteGroupMaxT][32];
  __shared__ int32_t s_flat[kRouteGroupMaxT * 32];  // ids [T, k]
  __shared__ int32_t s_cnt[258], s_off[258];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // The logits: the router's split partial sums added by every thread (all
  // loads in flight at once), or the finished rows copied.
  for (int q0 = tid; q0 < T * E1; q0 += 1024 * kSumCols) {
    float v[kSumCols];
    if (nsplit > 0) {
      sum_splits(part, nsplit, static_cast<size_t>(T) * E1, q0, 1024, T * E1, v);
    } else {
#pragma unroll
      for (int c = 0; c < kSumCols; ++c) {
        const int q = q0 + 1024 * c;
        v[c] = q < T * E1 ? logits[q] : 0.0f;
      }
    }
#pragma unroll
    for (int c = 0; c < kSumCols; ++c) {
      const int q = q0 + 1024 * c;
      if (q < T * E1) {
        s_lg[q] = v[c];
        if (nsplit > 0) logits[q] = v[c];  // [T, E1] rows read by later kernels
      }
    }
  }
  __syncthreads();
  if (warp < T) {
    topk_token_stage<8>(s_lg, nullptr, 0, warp, T, E, E1, k, norm_topk, ids, w, nullptr, s_ids[warp], s_sel[warp],
                        s_w[warp], nullptr);
    if (lane < k) s_flat[warp * k + lane] = s_ids[warp][lane];
  }
  __syncthreads();
  if constexpr (kWarp) {
    // few pairs: one warp groups them, every thread lists the tiles (one
    // barrier in between; the passes read only perm and the tile lists)
    small_group_schedule(s_flat, T, k, E, has_shared, perm, ctrl, I, Is, H, N, mt13, mt2, n13, n2, t13, t2);
  } else {
    group_stage(s_flat, T, k, E, has_shared, counts, offsets, perm, nullptr, 0, ctrl, s_cnt, s_off);
    __syncthreads();
    schedule_stage(s_cnt, s_off, E, I, Is, H, N, mt13, mt2, n13, n2, t13, t2);
  }
}

// Xs[pos, :] = x[token of perm[pos], :]: one warp per row, 16-byte chunks,
// up to 8 chunks per lane in flight.  Used for 17 to 32 tokens and past
// kFoldGatherMaxPairs pairs; in between the filing launch copies the rows.
__global__ void __launch_bounds__(256) tc_gather_kernel(const uint8_t* x, const int32_t* perm,
                                                        int P, int T, int k, int H, uint8_t* __restrict__ xs) {
  pdl_launch_dependents();  // let the next kernel on the stream launch early
  pdl_wait();               // inputs written by the previous kernel are visible
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * 8;
  const int nch = H >> 3;
  for (int pos = blockIdx.x * 8 + (threadIdx.x >> 5); pos < P; pos += warps) {
    const int p = perm[pos];
    const int t = p < T * k ? p / k : p - T * k;
    const uint8_t* src = x + static_cast<size_t>(t) * H * 2;
    uint8_t* dst = xs + static_cast<size_t>(pos) * H * 2;
    for (int c0 = lane; c0 < nch; c0 += 32 * 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + 32 * u < nch) v[u] = ld_nc16(src + 16 * (c0 + 32 * u));
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + 32 * u < nch) *reinterpret_cast<uint4*>(dst + 16 * (c0 + 32 * u)) = v[u];
    }
  }
}

// ================================================================ host
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D K-major map: `inner` elements per row (contiguous), `outer` rows of
// `row_stride` bytes; box of 64 x box_rows, 128-byte swizzle.
static bool make_map(CUtensorMap* m, int dtype, const void* base, uint64_t inner, uint64_t outer,
                     uint64_t row_stride, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_stride};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dtype == MOE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tc_shape_ok(const moe_cfg_t& c) {
  return (c.dtype == MOE_BF16 || c.dtype == MOE_F16) && c.hidden % 128 == 0 && c.inter % 64 == 0 &&
         c.shared_inter % 64 == 0;
}

bool tc_path_supported(const moe_cfg_t& c) { return tc_shape_ok(c) && encode_fn() != nullptr; }

template <int N, int MT>
static size_t tc_smem13() {
  constexpr uint32_t st = MT * kTileA + N * 128;
  constexpr int stg = 128 * 17 * 4;
  constexpr int ns = (kSmemBudget - stg) / st > 8 ? 8 : (kSmemBudget - stg) / st;
  return static_cast<size_t>(ns) * st + stg + 1024;
}
template <int N, int MT>
static size_t tc_smem2() {
  constexpr uint32_t st = MT * kTileA + 2 * N * 128;
  constexpr int ns = kSmemBudget / st > 8 ? 8 : kSmemBudget / st;
  return static_cast<size_t>(ns) * st + 1024;
}

// Two 128-row M-tiles per CTA: each token stage then feeds two accumulators.
constexpr int kMT = 2;

// M-tiles per W2 tile (1 or kMT).  Two share every activation stage (half the
// activation traffic); one spreads the weights over more CTAs, which only pays
// when it lowers the largest number of weight rows a CTA streams.  The
// distinct experts are unknown before the routing runs, so the count is taken
// at T*k experts (capped at E).
static int w2_m_tiles(int T, int k, int E, int H, int sms) {
  const int ex = (T * k < E ? T * k : E) + 1;  // with the shared expert
  const int t1 = ex * (H / 128), t2 = ex * ((H / 128 + kMT - 1) / kMT);
  // weight rows of the busiest CTA, in M-tiles: one M-tile per tile only if fewer
  return (t1 + sms - 1) / sms < kMT * ((t2 + sms - 1) / sms) ? 1 : kMT;
}

template <int DT, int N>
static moe_status_t launch_tc_passes(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws, const WsLayout& L,
                                     int32_t T, int fused_nsplit, cudaStream_t st) {
  const int H = c.hidden, E = c.n_experts, k = c.top_k, I = c.inter, Is = c.shared_inter;
  const int Imax = I > Is ? I : Is;
  const int P = static_cast<int>(L.pairs);
  Control* ctrl = reinterpret_cast<Control*>(ws + L.ctrl);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.g_counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.g_offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(ws + L.g_perm);
  int32_t* sched = reinterpret_cast<int32_t*>(ws + L.tc_sched);
  TcTile* t13 = reinterpret_cast<TcTile*>(ws + L.tc_tiles13);
  TcTile* t2 = reinterpret_cast<TcTile*>(ws + L.tc_tiles2);
  uint8_t* xs = ws + L.tc_xs;
  uint16_t* ahi = reinterpret_cast<uint16_t*>(ws + L.tc_act_hi);
  uint16_t* alo = reinterpret_cast<uint16_t*>(ws + L.tc_act_lo);
  float* y = reinterpret_cast<float*>(ws + L.g_y);
  const float* glog = reinterpret_cast<const float*>(ws + L.r_logits);
  const int gate_stride = c.has_shared_gate ? E + 1 : E;
  const uint64_t timeout = wait_timeout_ns();

  // M-tiles per W13 tile: two share every token stage (half the token
  // traffic), but when the pairs are few that leaves SMs idle, so a single
  // M-tile per CTA then spreads the weight stream over twice the SMs.
  const int sms0 = sm_count();
  const int est13 = (T * k < E ? T * k : E) * ((I / 64 + kMT - 1) / kMT);  // W13 tiles with kMT
  const int mt13 = est13 <= sms0 ? 1 : kMT;
  const int mt2 = w2_m_tiles(T, k, E, H, sms0);
  if (fused_nsplit >= 0) {  // ranking + grouping + tile lists in one launch (small batches)
    float* lg = reinterpret_cast<float*>(ws + L.r_logits);
    const int E1 = c.has_shared_gate ? E + 1 : E;
    const size_t lg_bytes = static_cast<size_t>(T) * E1 * sizeof(float);
    // the one-warp grouping wins up to T = 8 at k = 8 (measured); it needs the
    // pairs and the shared expert's entry within kWarpGroupPairs
    auto kern = T * k + (Is > 0 ? 1 : 0) <= kWarpGroupPairs ? route_group_kernel<true> : route_group_kernel<false>;
    if (raise_smem_limit(kern, lg_bytes) != cudaSuccess) return check_launch("route_group_kernel (smem)");
    launch_pdl(kern, dim3(1), dim3(1024), lg_bytes, st, lg, reinterpret_cast<const float*>(ws + L.r_part),
               fused_nsplit, T, E, E1, k, c.norm_topk, p.topk_ids, p.topk_w, Is > 0 ? 1 : 0, counts, offsets, perm,
               ctrl, I, Is, H, N, mt13, mt2, sched, sched + 1, t13, t2);
    if (moe_status_t s = check_launch("route_group_kernel")) return s;
  } else {  // pairs ranked by the top-k kernel
    int32_t* cnt = reinterpret_cast<int32_t*>(ws + L.tc_cnt);
    const int32_t* rank = reinterpret_cast<const int32_t*>(ws + L.tc_rank);
    // up to kFoldGatherMaxPairs pairs a warp per pair, copying the x rows too
    // (one 1024-thread CTA per SM); with more, the copy has a launch of its own
    // with twice the warps per SM
    const bool fold = P <= kFoldGatherMaxPairs;
    const int per = fold ? 32 : 1024;
    const int gq = (P + per - 1) / per;
    const int gf = 1 + (gq < sm_count() - 1 ? gq : sm_count() - 1);  // + CTA 0 for the tile lists
    launch_pdl(tc_fill_kernel, dim3(gf), dim3(1024), 0, st, p.topk_ids, rank, cnt, T, k, E,
               Is > 0 ? 1 : 0, perm, I, Is, H, N, mt13, mt2, sched, sched + 1, t13, t2,
               static_cast<const uint8_t*>(p.x), fold ? xs : nullptr, ctrl);
    if (moe_status_t s = check_launch("tc_fill_kernel")) return s;
  }
  const int sms = sm_count();
  // Up to 16 tokens the W13 pass reads x itself (B = all T tokens, each pair
  // takes its token's accumulator column) and the gather of x rows into expert
  // order is not needed (T = 2 / 8 / 16: about 2 us less per layer).  With
  // more tokens every CTA reads the same x rows at the same time (8 KB per
  // stage at T = 64, +10 us per layer), so the gathered rows are used.
  const bool direct = T <= 16 && T <= N;
  const bool gather = !direct && (fused_nsplit >= 0 || P > kFoldGatherMaxPairs);
  if (gather) {
    const int gg = (P + 7) / 8 < sms * 8 ? (P + 7) / 8 : sms * 8;
    launch_pdl(tc_gather_kernel, dim3(gg), dim3(256), 0, st, static_cast<const uint8_t*>(p.x), perm, P, T, k, H, xs);
    if (moe_status_t s = check_launch("tc_gather_kernel")) return s;
  }

  CUtensorMap mA, mAs, mB, mW2, mW2s, mHi, mLo, mHiS, mLoS;
  const void* sw13 = p.shared_w13 ? p.shared_w13 : p.w13;
  const void* sw2 = p.shared_w2 ? p.shared_w2 : p.w2;
  const int IsM = Is > 0 ? Is : I;
  bool ok = make_map(&mA, DT, p.w13, H, static_cast<uint64_t>(E) * 2 * I, static_cast<uint64_t>(H) * 2, 64) &&
            make_map(&mAs, DT, sw13, H, 2ull * IsM, static_cast<uint64_t>(H) * 2, 64) &&
            (direct ? make_map(&mB, DT, p.x, H, T, static_cast<uint64_t>(H) * 2, N)
                    : make_map(&mB, DT, xs, H, P, static_cast<uint64_t>(H) * 2, N)) &&
            make_map(&mW2, DT, p.w2, I, static_cast<uint64_t>(E) * H, static_cast<uint64_t>(I) * 2, 128) &&
            make_map(&mW2s, DT, sw2, IsM, H, static_cast<uint64_t>(IsM) * 2, 128) &&
            make_map(&mHi, DT, ahi, I, P, static_cast<uint64_t>(Imax) * 2, N) &&
            make_map(&mLo, DT, alo, I, P, static_cast<uint64_t>(Imax) * 2, N) &&
            make_map(&mHiS, DT, ahi, IsM, P, static_cast<uint64_t>(Imax) * 2, N) &&
            make_map(&mLoS, DT, alo, IsM, P, static_cast<uint64_t>(Imax) * 2, N);
  if (!ok) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed");

  const int g13 = static_cast<int>(L.tc_max13 < sms ? L.tc_max13 : sms);
  const int g2 = static_cast<int>(L.tc_max2 < sms ? L.tc_max2 : sms);
  auto launch13 = [&](auto kernel, size_t s13) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s13));
    launch_pdl(kernel, dim3(g13 > 0 ? g13 : 1), dim3(kTcThreads), s13, st, mA, mAs, mB, t13, sched, H, I, Is, E,
               Imax, ahi, alo, ctrl, timeout, perm, direct ? T : 0, k, sched + 2,
               fused_nsplit >= 0 ? nullptr : reinterpret_cast<int32_t*>(ws + L.tc_cnt), E);
  };
  if (mt13 == 1) {
    if (direct) launch13(tc_w13_kernel<DT, N, 1, true>, tc_smem13<N, 1>());
    else launch13(tc_w13_kernel<DT, N, 1, false>, tc_smem13<N, 1>());
  } else {
    if (direct) launch13(tc_w13_kernel<DT, N, kMT, true>, tc_smem13<N, kMT>());
    else launch13(tc_w13_kernel<DT, N, kMT, false>, tc_smem13<N, kMT>());
  }
  if (moe_status_t s = check_launch("tc_w13_kernel")) return s;
  auto launch2 = [&](auto kernel, size_t s2) {
    cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(s2));
    launch_pdl(kernel, dim3(g2 > 0 ? g2 : 1), dim3(kTcThreads), s2, st, mW2, mW2s, mHi, mLo, mHiS, mLoS, t2,
               sched + 1, perm, p.topk_w, glog, gate_stride, c.has_shared_gate, T, H, I, Is, E, k, y, sched + 3, ctrl,
               timeout);
  };
  if (mt2 == 1) launch2(tc_w2_kernel<DT, N, 1>, tc_smem2<N, 1>());
  else launch2(tc_w2_kernel<DT, N, kMT>, tc_smem2<N, kMT>());
  if (moe_status_t s = check_launch("tc_w2_kernel")) return s;
  stat_kernels(gather ? 4 : 3);
  return MOE_OK;
}


bool tc_router_supported(const moe_cfg_t& c) {
  return (c.dtype == MOE_BF16 || c.dtype == MOE_F16) && c.hidden % 64 == 0 && encode_fn() != nullptr;
}

// logits [T, E1] (E1 = E, or E + 1 with the gate column) on tensor cores.
moe_status_t launch_tc_router(const moe_cfg_t& c, const void* x, const void* router_w, const void* gate_w,
                              int32_t T, float* logits, float* part, int E1, Control* ctrl, cudaStream_t st,
                              int* nsplit) {
  constexpr int N = 128;
  const int DT = c.dtype;
  const int H = c.hidden, E = c.n_experts;
  const int mE = (E + 127) / 128;
  const int nm = mE + (gate_w ? 1 : 0);
  CUtensorMap mWr, mG, mX;
  bool ok = make_map(&mWr, DT, router_w, H, E, static_cast<uint64_t>(H) * 2, 128) &&
            make_map(&mG, DT, gate_w ? gate_w : router_w, H, 1, static_cast<uint64_t>(H) * 2, 128) &&
            make_map(&mX, DT, x, H, T, static_cast<uint64_t>(H) * 2, N);
  if (!ok) return set_error(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (router)");
  constexpr uint32_t st_bytes = kTileA + N * 128;
  constexpr int ns = kSmemBudget / st_bytes > 8 ? 8 : kSmemBudget / st_bytes;
  const size_t smem = static_cast<size_t>(ns) * st_bytes + 1024;
  auto kern = DT == MOE_BF16 ? tc_router_kernel<MOE_BF16, N> : tc_router_kernel<MOE_F16, N>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  const int tiles0 = nm * ((T + N - 1) / N);
  const int sms = sm_count();
  // K splits when the tiles would leave most SMs idle (T = 512: 12 tiles, 5.4
  // us less per layer; at T = 4096, 96 tiles, four splits cost 4 us in partial
  // sums): the fewest rounds of (K blocks per split + 2 for the epilogue)
  int S = 1;
  if (part && E <= 256 && 2 * tiles0 <= sms) {
    int best = 1 << 30;
    for (int sp = 1; sp <= kRouterMaxSplits && (H / kBK) % sp == 0; sp *= 2) {
      const int cost = ((tiles0 * sp + sms - 1) / sms) * (H / kBK / sp + 2);
      if (cost < best) { best = cost; S = sp; }
    }
  }
  *nsplit = S > 1 ? S : 0;
  const int tiles = tiles0 * S;
  const int g = tiles < sms ? tiles : sms;
  launch_pdl(kern, dim3(g), dim3(kTcThreads), smem, st, mWr, mG, mX, T, H, E, E1, mE, nm, S,
             S > 1 ? part : logits, ctrl, wait_timeout_ns());
  if (moe_status_t s = check_launch("tc_router_kernel")) return s;
  stat_kernels(1);
  return MOE_OK;
}

int tc_tile_n(const moe_cfg_t& c, int32_t T) {
  const double avg = static_cast<double>(T) * c.top_k / c.n_experts;
  return avg > 48.0 ? 128 : 64;
}

moe_status_t launch_tc_passes(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws, const WsLayout& L, int32_t T,
                              int fused_nsplit, cudaStream_t st) {
  if (c.dtype == MOE_BF16) {
    if (L.tc_n == 128) return launch_tc_passes<MOE_BF16, 128>(c, p, ws, L, T, fused_nsplit, st);
    return launch_tc_passes<MOE_BF16, 64>(c, p, ws, L, T, fused_nsplit, st);
  }
  if (L.tc_n == 128) return launch_tc_passes<MOE_F16, 128>(c, p, ws, L, T, fused_nsplit, st);
  return launch_tc_passes<MOE_F16, 64>(c, p, ws, L, T, fused_nsplit, st);
}

}  // namespace moe
