// moe_api.cu — the library's extern "C" entry points (declared in moe.h):
// argument validation, workspace layout, dispatch to the kernels, error
// text, path counters and the device status word.

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

// ------------------------------------------------------------------ errors
static thread_local char g_err[512] = "";

moe_status_t set_error(moe_status_t code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

moe_status_t check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return MOE_OK;
}

// ---------------------------------------------------------------- counters
static std::atomic<uint64_t> g_decode{0}, g_router{0}, g_grouped{0}, g_grouped_tc{0}, g_kernels{0},
    g_decode_general{0};
void stat_decode() { g_decode.fetch_add(1, std::memory_order_relaxed); }
void stat_decode_general() { g_decode_general.fetch_add(1, std::memory_order_relaxed); }
void stat_router() { g_router.fetch_add(1, std::memory_order_relaxed); }
void stat_grouped() { g_grouped.fetch_add(1, std::memory_order_relaxed); }
void stat_grouped_tc() { g_grouped_tc.fetch_add(1, std::memory_order_relaxed); }
void stat_kernels(uint64_t n) { g_kernels.fetch_add(n, std::memory_order_relaxed); }

// ------------------------------------------------------------ device facts
int sm_count() {
  static int cached[64];
  static bool have[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!have[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    cached[dev] = n;
    have[dev] = true;
  }
  return cached[dev];
}

static std::atomic<uint64_t> g_timeout_ns{2000000000ull};

std::mutex& attr_mutex() {
  static std::mutex mu;
  return mu;
}
uint64_t wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

// ---------------------------------------------------------- workspace layout
WsLayout ws_layout(const moe_cfg_t& c, int32_t T) {
  WsLayout L;
  const int64_t H = c.hidden, E = c.n_experts, k = c.top_k, I = c.inter, Is = c.shared_inter;
  size_t off = sizeof(Control);
  L.ctrl = 0;
  L.ll_logits = off;
  off = align_up(off + kLogitReplicas * ((E + 2) & ~int64_t(1)) * 8, kWsAlign);
  L.ll_act = off;
  off = align_up(off + kActReplicas * ((k * I + Is + 1) & ~int64_t(1)) * 8, kWsAlign);
  L.r_logits = off;
  off = align_up(off + static_cast<size_t>(T) * (E + 1) * 4, kWsAlign);
  L.r_part = off;
  if (T <= 64) {
    off = align_up(off + static_cast<size_t>(H / 256 + 1) * T * (E + 1) * 4, kWsAlign);
  } else if (T >= kRouterTcMinT && E <= 256) {  // the tensor-core router's K-split partial sums
    L.r_part_splits = kRouterMaxSplits;
    off = align_up(off + static_cast<size_t>(kRouterMaxSplits) * T * (E + 1) * 4, kWsAlign);
  }
  if (T > 1) {
    const int64_t P = T * k + (Is > 0 ? T : 0);
    const int64_t tn = 8;  // pairs per tile of the grouped kernels
    L.pairs = P;
    L.max_tiles = (T * k + tn - 1) / tn + E + (Is > 0 ? (T + tn - 1) / tn : 0) + 1;
    L.g_counts = off;
    off = align_up(off + (E + 2) * 4, kWsAlign);
    L.g_offsets = off;
    off = align_up(off + (E + 2) * 4, kWsAlign);
    L.g_perm = off;
    off = align_up(off + P * 4, kWsAlign);
    L.g_tiles = off;
    off = align_up(off + (L.max_tiles + 1) * 8, kWsAlign);
    L.g_act = off;
    off = align_up(off + static_cast<size_t>(P) * (I > Is ? I : Is) * 4, kWsAlign);
    L.g_y = off;
    off = align_up(off + static_cast<size_t>(P) * H * 4, kWsAlign);
    if (tc_shape_ok(c)) {
      const int64_t N = tc_tile_n(c, T);
      const int64_t nt_routed = (T * k + N - 1) / N + E;
      const int64_t nt_shared = Is > 0 ? (T + N - 1) / N : 0;
      L.tc_n = static_cast<int>(N);
      L.tc_max13 = nt_routed * (I / 64) + nt_shared * (Is / 64);
      L.tc_max2 = (nt_routed + nt_shared) * (H / 128);
      L.tc_sched = off;
      off = align_up(off + 16, kWsAlign);
      L.tc_tiles13 = off;
      off = align_up(off + static_cast<size_t>(L.tc_max13) * 16, kWsAlign);
      L.tc_tiles2 = off;
      off = align_up(off + static_cast<size_t>(L.tc_max2) * 16, kWsAlign);
      L.tc_xs = off;
      off = align_up(off + static_cast<size_t>(P) * H * 2, kWsAlign);
      L.tc_cnt = off;
      off = align_up(off + static_cast<size_t>(E) * 4, kWsAlign);
      L.tc_rank = off;
      off = align_up(off + static_cast<size_t>(T) * k * 4, kWsAlign);
      const int64_t Imax = I > Is ? I : Is;
      L.tc_act_hi = off;
      off = align_up(off + static_cast<size_t>(P) * Imax * 2, kWsAlign);
      L.tc_act_lo = off;
      off = align_up(off + static_cast<size_t>(P) * Imax * 2, kWsAlign);
    }
  }
  if (batch_ws_shape_ok(c, T)) {
    size_t lw, aw;
    const size_t pw = batch_ws_words(c, T, lw, aw);
    L.bt_logits = off;
    off = align_up(off + lw * 8, kWsAlign);
    L.bt_act = off;
    off = align_up(off + aw * 8, kWsAlign);
    L.bt_part = off;
    off = align_up(off + pw * 8, kWsAlign);
  }
  L.total = off;
  return L;
}

// -------------------------------------------------------------- validation
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static moe_status_t check_cfg(const moe_cfg_t* c) {
  if (!c) return set_error(MOE_ERR_INVALID_ARG, "cfg is NULL");
  if (c->hidden <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->inter <= 0 || c->shared_inter < 0)
    return set_error(MOE_ERR_INVALID_ARG, "cfg: sizes must be positive (shared_inter >= 0)");
  if (c->dtype != MOE_F16 && c->dtype != MOE_BF16)
    return set_error(MOE_ERR_UNSUPPORTED, "cfg: dtype must be MOE_F16 or MOE_BF16");
  if (c->out_dtype != c->dtype && c->out_dtype != MOE_F32)
    return set_error(MOE_ERR_UNSUPPORTED, "cfg: out_dtype must equal dtype or be MOE_F32");
  if (c->norm_topk != 0 && c->norm_topk != 1) return set_error(MOE_ERR_INVALID_ARG, "cfg: norm_topk is 0 or 1");
  if (c->has_shared_gate != 0 && c->has_shared_gate != 1)
    return set_error(MOE_ERR_INVALID_ARG, "cfg: has_shared_gate is 0 or 1");
  if (c->has_shared_gate && c->shared_inter == 0)
    return set_error(MOE_ERR_INVALID_ARG, "cfg: a shared gate needs a shared expert");
  if (c->flags & ~(MOE_FLAG_GROUPED_SIMT | MOE_FLAG_GROUPED_TC | MOE_FLAG_STATIC_WEIGHTS | MOE_FLAG_RESIDUAL |
                   MOE_FLAG_GROUPED_SINGLE))
    return set_error(MOE_ERR_INVALID_ARG, "cfg: unknown flag bits");
  {
    const int path = c->flags & (MOE_FLAG_GROUPED_SIMT | MOE_FLAG_GROUPED_TC | MOE_FLAG_GROUPED_SINGLE);
    if (path & (path - 1))
      return set_error(MOE_ERR_INVALID_ARG,
                       "cfg: MOE_FLAG_GROUPED_SIMT, MOE_FLAG_GROUPED_TC and MOE_FLAG_GROUPED_SINGLE exclude each other");
  }
  if (c->hidden % 8 || c->inter % 8 || c->shared_inter % 8)
    return set_error(MOE_ERR_UNSUPPORTED, "cfg: hidden, inter and shared_inter must be multiples of 8");
  if (c->top_k > 32 || c->top_k > c->n_experts)
    return set_error(MOE_ERR_UNSUPPORTED, "cfg: top_k must be <= 32 and <= n_experts");
  if (c->n_experts > 1024) return set_error(MOE_ERR_UNSUPPORTED, "cfg: n_experts must be <= 1024");
  return MOE_OK;
}

static moe_status_t check_ptr(const void* p, const char* name) {
  if (!p) return set_error(MOE_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return set_error(MOE_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return MOE_OK;
}

moe_status_t check_ws(const moe_cfg_t& c, const void* ws, size_t ws_bytes, int32_t T, WsLayout& L) {
  L = ws_layout(c, T);
  if (!ws) return set_error(MOE_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", L.total);
  if (reinterpret_cast<uintptr_t>(ws) % kWsAlign)
    return set_error(MOE_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < L.total)
    return set_error(MOE_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", ws_bytes, L.total);
  return MOE_OK;
}

moe_status_t check_block(const moe_cfg_t* c, const void* x, const void* router_w, const void* w13,
                         const void* w2, const void* sw13, const void* sw2, const void* swg, moe_topk_t topk,
                         const void* out) {
  if (moe_status_t s = check_cfg(c)) return s;
  if (moe_status_t s = check_ptr(x, "x")) return s;
  if (moe_status_t s = check_ptr(router_w, "router_w")) return s;
  if (moe_status_t s = check_ptr(w13, "w13")) return s;
  if (moe_status_t s = check_ptr(w2, "w2")) return s;
  if (moe_status_t s = check_ptr(out, "out")) return s;
  if (!topk.ids || !topk.weights) return set_error(MOE_ERR_INVALID_ARG, "topk.ids / topk.weights is NULL");
  if (c->shared_inter > 0) {
    if (moe_status_t s = check_ptr(sw13, "shared_w13")) return s;
    if (moe_status_t s = check_ptr(sw2, "shared_w2")) return s;
  } else if (sw13 || sw2) {
    return set_error(MOE_ERR_INVALID_ARG, "shared weights given but shared_inter == 0");
  }
  if (c->has_shared_gate) {
    if (moe_status_t s = check_ptr(swg, "shared_gate_w")) return s;
  } else if (swg) {
    return set_error(MOE_ERR_INVALID_ARG, "shared_gate_w given but has_shared_gate == 0");
  }
  if (out == x) return set_error(MOE_ERR_INVALID_ARG, "out must not alias x");
  return MOE_OK;
}

// --------------------------------------------------------------- test hook
__global__ void wait_test_kernel(Control* ctrl, uint64_t timeout_ns) {
  const uint64_t deadline = global_ns() + timeout_ns;
  while (ld_relaxed_u32(&ctrl->never_set) == 0u) {
    if (global_ns() > deadline) {
      report_error(ctrl, kDevTimeoutTest, blockIdx.x);
      return;
    }
  }
}

moe_status_t launch_wait_test(uint8_t* ws, cudaStream_t st) {
  wait_test_kernel<<<1, 1, 0, st>>>(reinterpret_cast<Control*>(ws), wait_timeout_ns());
  if (moe_status_t s = check_launch("wait_test_kernel")) return s;
  stat_kernels(1);
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

size_t moe_workspace_bytes(const moe_cfg_t* cfg, int32_t T) {
  if (check_cfg(cfg) != MOE_OK || T < 1) return 0;
  return ws_layout(*cfg, T).total;
}

moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < sizeof(Control)) return set_error(MOE_ERR_WORKSPACE, "workspace NULL or too small");
  if (cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return check_launch("cudaMemsetAsync(workspace)");
  return MOE_OK;
}

moe_status_t moe_router_topk(const moe_cfg_t* cfg, const void* x, const void* router_w, int32_t T,
                             moe_topk_t topk, float* logits, void* ws, size_t ws_bytes, void* stream) {
  if (moe_status_t s = check_cfg(cfg)) return s;
  if (T < 0) return set_error(MOE_ERR_INVALID_ARG, "T must be >= 0");
  if (T == 0) return MOE_OK;  // nothing to do; the per-token buffers may be empty (NULL)
  if (moe_status_t s = check_ptr(x, "x")) return s;
  if (moe_status_t s = check_ptr(router_w, "router_w")) return s;
  if (!topk.ids || !topk.weights) return set_error(MOE_ERR_INVALID_ARG, "topk.ids / topk.weights is NULL");
  WsLayout L;
  if (moe_status_t s = check_ws(*cfg, ws, ws_bytes, T, L)) return s;
  // The router-only entry ranks the E routed experts; the gate column is not needed.
  moe_cfg_t c = *cfg;
  c.has_shared_gate = 0;
  if (moe_status_t s = launch_router(c, x, router_w, nullptr, T, topk.ids, topk.weights, logits,
                                     static_cast<uint8_t*>(ws), L, static_cast<cudaStream_t>(stream)))
    return s;
  stat_router();
  return MOE_OK;
}

moe_status_t moe_decode_forward(const moe_cfg_t* cfg, const void* x, const void* router_w, const void* w13,
                                const void* w2, const void* shared_w13, const void* shared_w2,
                                const void* shared_gate_w, moe_topk_t topk, void* out, void* ws,
                                size_t ws_bytes, void* stream) {
  if (moe_status_t s = check_block(cfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, topk, out))
    return s;
  WsLayout L;
  if (moe_status_t s = check_ws(*cfg, ws, ws_bytes, 1, L)) return s;
  BlockPtrs p{x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, topk.ids, topk.weights, out};
  if (moe_status_t s = launch_decode_fused(*cfg, p, static_cast<uint8_t*>(ws), L, static_cast<cudaStream_t>(stream)))
    return s;
  stat_decode();
  return MOE_OK;
}

moe_status_t moe_grouped_forward(const moe_cfg_t* cfg, const void* x, const void* router_w, const void* w13,
                                 const void* w2, const void* shared_w13, const void* shared_w2,
                                 const void* shared_gate_w, moe_topk_t topk, void* out, void* ws,
                                 size_t ws_bytes, int32_t T, void* stream) {
  if (T < 0) return set_error(MOE_ERR_INVALID_ARG, "T must be >= 0");
  if (T == 0) return check_cfg(cfg);  // nothing to do; the per-token buffers may be empty (NULL)
  if (moe_status_t s = check_block(cfg, x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, topk, out))
    return s;
  WsLayout L;
  if (moe_status_t s = check_ws(*cfg, ws, ws_bytes, T, L)) return s;
  BlockPtrs p{x, router_w, w13, w2, shared_w13, shared_w2, shared_gate_w, topk.ids, topk.weights, out};
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 1) {
    if (moe_status_t s = launch_decode_fused(*cfg, p, static_cast<uint8_t*>(ws), L, st)) return s;
    stat_decode();
    return MOE_OK;
  }
  if (static_cast<int64_t>(T) * cfg->top_k > (1 << 30))
    return set_error(MOE_ERR_UNSUPPORTED, "T * top_k too large");
  // 2 <= T <= 16: the single-launch kernel when asked for, or by default when
  // the shape allows it and no other T > 1 path was asked for: up to 8 tokens
  // (3 when I < 256: its W2 units of 16 short rows are copy-issue-bound there),
  // and up to 16 where the tensor-core passes are not available.  Measured:
  // I = 512, from 9 tokens the tensor-core passes are faster; I = 128 (fp16),
  // T = 2 / 4 / 8: 22.1 / 32.8 / 52.2 us against 28.4 / 31.6 / 40.2 there.
  const bool other = cfg->flags & (MOE_FLAG_GROUPED_SIMT | MOE_FLAG_GROUPED_TC);
  const int single_max = cfg->inter >= 256 ? 8 : 3;
  const bool single_default =
      !other && batch_shape_ok(*cfg, T) && (T <= single_max || !tc_path_supported(*cfg));
  if ((cfg->flags & MOE_FLAG_GROUPED_SINGLE) || single_default) {
    if (moe_status_t s = launch_decode_batch(*cfg, p, static_cast<uint8_t*>(ws), L, T, st)) return s;
    stat_grouped();
    return MOE_OK;
  }
  if (moe_status_t s = launch_grouped(*cfg, p, static_cast<uint8_t*>(ws), L, T, st)) return s;
  stat_grouped();
  return MOE_OK;
}

moe_status_t moe_query_status(void* ws, void* stream) {
  if (!ws) {
    // The allocation-free entry keeps its status word in its built-in array.
    if (moe_status_t s = noalloc_scratch(&ws)) return s;
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return check_launch("cudaStreamSynchronize");
  uint32_t hdr[2] = {0, 0};
  if (cudaMemcpy(hdr, ws, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess)
    return check_launch("cudaMemcpy(status)");
  if (hdr[0] == kDevOk) return MOE_OK;
  const uint32_t zero[2] = {0, 0};
  if (cudaMemcpy(ws, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return check_launch("cudaMemcpy(clear status)");
  static const char* names[] = {"ok", "timeout waiting for router logits", "timeout waiting for activations",
                                "timeout waiting for a bulk copy", "expert id out of range",
                                "test wait ran out"};
  const char* what = hdr[0] < 6 ? names[hdr[0]] : "unknown";
  if (hdr[0] == kDevBadExpert)
    return set_error(MOE_ERR_DEVICE, "device check: %s (pair %u)", what, hdr[1]);
  return set_error(MOE_ERR_TIMEOUT, "device wait: %s (CTA %u)", what, hdr[1]);
}

const char* moe_last_error(void) { return g_err; }

moe_status_t moe_get_stats(moe_stats_t* stats) {
  if (!stats) return set_error(MOE_ERR_INVALID_ARG, "stats is NULL");
  stats->decode_fused_calls = g_decode.load();
  stats->router_calls = g_router.load();
  stats->grouped_calls = g_grouped.load();
  stats->grouped_tc_calls = g_grouped_tc.load();
  stats->kernels_launched = g_kernels.load();
  stats->decode_general_calls = g_decode_general.load();
  return MOE_OK;
}

void moe_reset_stats(void) {
  g_decode = 0;
  g_router = 0;
  g_grouped = 0;
  g_grouped_tc = 0;
  g_kernels = 0;
  g_decode_general = 0;
}

moe_status_t moe_set_wait_timeout_ns(uint64_t ns) {
  if (ns < 1000) return set_error(MOE_ERR_INVALID_ARG, "timeout below 1000 ns");
  g_timeout_ns.store(ns);
  return MOE_OK;
}

moe_status_t moe_test_wait_timeout(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < sizeof(Control)) return set_error(MOE_ERR_WORKSPACE, "workspace NULL or too small");
  if (reinterpret_cast<uintptr_t>(ws) % kWsAlign) return set_error(MOE_ERR_WORKSPACE, "workspace not 256-B aligned");
  return launch_wait_test(static_cast<uint8_t*>(ws), static_cast<cudaStream_t>(stream));
}

}  // extern "C"
