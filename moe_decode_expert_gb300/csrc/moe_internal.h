// moe_internal.h — host-side plumbing shared by the library's translation
// units: workspace layout, launch helpers, error reporting and counters.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "moe.h"

namespace moe {

constexpr size_t kWsAlign = 256;
// Copies of the router-logit exchange words of the single-launch decode (each
// CTA reads one copy, so fewer CTAs poll each L2 line): the most any
// instantiation writes (the workspace holds this many).
constexpr int kLogitReplicas = 16;
// Copies of the activation exchange words (each CTA reads one copy): the most.
constexpr int kActReplicas = 8;
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
// Most tokens of the single-launch batch kernel (2 <= T <= kBatchMaxT).
constexpr int kBatchMaxT = 16;

// Byte offsets of every region of one workspace, for `T` tokens of a cfg.
struct WsLayout {
  size_t ctrl = 0;        // Control block, 256 B
  // single-launch decode (T == 1): exchange words between CTAs
  size_t ll_logits = 0;   // kLogitReplicas x (E + 1) words of 8 B, each copy padded to even
  size_t ll_act = 0;      // kActReplicas x (k*I + Is) words, each copy padded to even
  // router for T tokens
  size_t r_logits = 0;    // [T, E + 1] fp32 (column E: shared-gate logit)
  size_t r_part = 0;      // T <= 64: [H / 256 + 1, T, E + 1] fp32 split partial logits;
                          // T >= kRouterTcMinT: [r_part_splits, T, E + 1] (tensor-core router)
  int r_part_splits = 0;  // K splits the tensor-core router may use (0: none)
  // grouped path (T > 1)
  size_t g_counts = 0;    // (E + 2) int32: tokens per expert (E = shared)
  size_t g_offsets = 0;   // (E + 2) int32: exclusive prefix of counts
  size_t g_perm = 0;      // [P] int32: pair ids grouped by expert
  size_t g_tiles = 0;     // [max_tiles + 1] int32 x2: (expert, first row) per tile
  size_t g_act = 0;       // [P, max(I, Is)] fp32
  size_t g_y = 0;         // [P, H] fp32 weighted expert outputs
  // tensor-core grouped path (T > 1, bf16, H % 128 == 0, I and Is % 64 == 0)
  size_t tc_sched = 0;    // 2 int32: tile counts of the two passes
  size_t tc_tiles13 = 0;  // [tc_max13] tiles of the W13 pass
  size_t tc_tiles2 = 0;   // [tc_max2] tiles of the W2 pass
  size_t tc_xs = 0;       // [P, H] x rows gathered in expert order
  size_t tc_cnt = 0;      // [E] int32 pair counters (zero between calls) of the ranked grouping
  size_t tc_rank = 0;     // [T * k] int32: each pair's rank within its expert
  size_t tc_act_hi = 0;   // [P, max(I, Is)] activation, leading term
  size_t tc_act_lo = 0;   // [P, max(I, Is)] activation, remainder term
  // single-launch batch kernel (2 <= T <= kBatchMaxT): exchange words
  size_t bt_logits = 0;   // kLogitReplicas x [T][E + 1 padded to even] words
  size_t bt_act = 0;      // [T*k + 1 slots][T][max(I, Is)] words (slot T*k: shared expert)
  size_t bt_part = 0;     // [T*k + 1 slots][T][H] words
  int tc_n = 0;           // tokens per tile (0 = path not laid out)
  int64_t tc_max13 = 0;
  int64_t tc_max2 = 0;
  size_t total = 0;
  int64_t pairs = 0;      // P = T*k + (Is ? T : 0)
  int64_t max_tiles = 0;
};

WsLayout ws_layout(const moe_cfg_t& c, int32_t T);

// Host-side validation of one block call's arguments (cfg, pointers,
// aliasing) and of a workspace for T tokens (fills L).  No CUDA call.
moe_status_t check_block(const moe_cfg_t* c, const void* x, const void* router_w, const void* w13,
                         const void* w2, const void* sw13, const void* sw2, const void* swg, moe_topk_t topk,
                         const void* out);
moe_status_t check_ws(const moe_cfg_t& c, const void* ws, size_t ws_bytes, int32_t T, WsLayout& L);

// Device address of the allocation-free entry's built-in scratch array on the
// current device (looked up once per device), for moe_query_status(NULL).
moe_status_t noalloc_scratch(void** out);

// Host-side error recording (thread-local text + code).
moe_status_t set_error(moe_status_t code, const char* fmt, ...);
moe_status_t check_launch(const char* what);

// Process-wide counters.
void stat_decode();
void stat_decode_general();
void stat_router();
void stat_grouped();
void stat_grouped_tc();
void stat_kernels(uint64_t n);

// Device properties cached per device.
int sm_count();
uint64_t wait_timeout_ns();

// Pointers of one MoE block call.
struct BlockPtrs {
  const void* x;
  const void* router_w;
  const void* w13;
  const void* w2;
  const void* shared_w13;
  const void* shared_w2;
  const void* shared_gate_w;
  int32_t* topk_ids;
  float* topk_w;
  void* out;
};

// Kernel launchers (each returns MOE_OK or a host-side error).
moe_status_t launch_decode_fused(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws,
                                 const WsLayout& L, cudaStream_t st);
// With nsplit_out != NULL the top-k launch is skipped and *nsplit_out tells
// how the logits were left (split partial sums, or 0: plain [T, E1] rows).
// With cnt != NULL the top-k kernel also ranks every pair within its expert:
// rank[t * k + j] = atomicAdd(&cnt[ids[t * k + j]], 1) (cnt zero beforehand).
moe_status_t launch_router(const moe_cfg_t& c, const void* x, const void* router_w,
                           const void* shared_gate_w, int32_t T, int32_t* ids, float* w,
                           float* logits_out, uint8_t* ws, const WsLayout& L, cudaStream_t st,
                           int* nsplit_out = nullptr, int32_t* cnt = nullptr, int32_t* rank = nullptr);
moe_status_t launch_grouped(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws, const WsLayout& L,
                            int32_t T, cudaStream_t st);
moe_status_t launch_wait_test(uint8_t* ws, cudaStream_t st);

// Single-launch kernel for 2 <= T <= kBatchMaxT (moe_batch.cu).
// batch_ws_shape_ok: the shape conditions that lay out its workspace regions
// (no CUDA call); batch_shape_ok: those plus the grid and shared-memory fit
// on the current device.
bool batch_ws_shape_ok(const moe_cfg_t& c, int32_t T);
bool batch_shape_ok(const moe_cfg_t& c, int32_t T);
// Exchange words of the batch kernel: returns the partial words; sets the
// logit and activation word counts.
size_t batch_ws_words(const moe_cfg_t& c, int32_t T, size_t& logit_words, size_t& act_words);
moe_status_t launch_decode_batch(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws, const WsLayout& L,
                                 int32_t T, cudaStream_t st);

// Tensor-core grouped passes (moe_grouped_tc.cu).
bool tc_shape_ok(const moe_cfg_t& c);        // shape/dtype eligibility (host only)
bool tc_path_supported(const moe_cfg_t& c);  // eligibility and the TMA encoder is available
int tc_tile_n(const moe_cfg_t& c, int32_t T);
struct Control;
bool tc_router_supported(const moe_cfg_t& c);
// part: room for kRouterMaxSplits x [T, E1] fp32 partial sums, or NULL (no
// K split); *nsplit: the splits left in part (0: the logits are in `logits`).
constexpr int kRouterMaxSplits = 8;
constexpr int kRouterTcMinT = 256;  // bf16 and T from this on: tensor-core router
moe_status_t launch_tc_router(const moe_cfg_t& c, const void* x, const void* router_w, const void* gate_w,
                              int32_t T, float* logits, float* part, int E1, Control* ctrl, cudaStream_t st,
                              int* nsplit);
// fused_nsplit >= 0: the router ran without its top-k (logits as that many
// split partial sums, 0 = plain); ranking, grouping and the tile lists then run
// as one launch.  -1: ids and the grouping are already in the workspace.
moe_status_t launch_tc_passes(const moe_cfg_t& c, const BlockPtrs& p, uint8_t* ws, const WsLayout& L, int32_t T,
                              int fused_nsplit, cudaStream_t st);

// Serialises every read-then-raise of a kernel attribute (any host thread).
std::mutex& attr_mutex();

// Raise, never lower, a kernel's dynamic shared-memory limit on the current
// device: a graph captured with a larger launch still runs after a call that
// needed less.  The check and the set run under one process-wide lock, so two
// host threads cannot interleave them and lower a limit the other just set.
template <typename K>
inline cudaError_t raise_smem_limit(K kernel, size_t bytes) {
  std::lock_guard<std::mutex> lock(attr_mutex());
  cudaFuncAttributes fa;
  cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return e;
  if (static_cast<size_t>(fa.maxDynamicSharedSizeBytes) >= bytes) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel on the stream drains.  Every kernel of the library
// runs griddepcontrol.wait before it reads anything an earlier kernel may
// write (only set-up that reads no such memory — barrier initialisation, TMEM
// allocation, tensor-map prefetch, weight loads with static weights — may come
// first), and those reads are loads the compiler cannot move above the wait,
// so ordering is unchanged; only the launch latency overlaps.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

#ifdef MOE_PHASE_TRACE
// Trace build: the stamp record of the next T = 1 launch (ring of launches).
uint64_t* trace_next_record();
#endif

// Grid size of the single-launch decode kernel for cfg c.
int decode_grid(const moe_cfg_t& c);
// Dynamic shared memory of that kernel (bytes) for grid G.
size_t decode_smem_bytes(const moe_cfg_t& c, int G);

}  // namespace moe
