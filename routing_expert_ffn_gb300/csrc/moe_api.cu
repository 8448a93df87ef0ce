// C ABI of libmoe.so: argument checks, workspace layout, and the launch
// sequence of the routed-expert MoE path.  See include/moe.h for the contract.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// One status word per device, shared by every call on that device.
static __device__ unsigned g_status_word;

// Scratch of moe_dispatch_static_scratch (the one entry point without a
// workspace): a file-scope device array, so every GPU that loads the library
// holds these bytes until the process exits.
constexpr size_t kStaticDispatchScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_dispatch_scratch[kStaticDispatchScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
// Condensation walks a bucket's representatives as a shared-memory bitset of up to 65536
// rows; a bucket holds each token at most once, so T <= 65536 bounds every bucket.
constexpr int kCondenseMaxTokens = 65536;

// Device addresses of the two file-scope arrays (in host code their names are only
// host-side stand-ins, never device addresses) and the SM count.
struct DeviceInfo {
  int num_sms = 0;
  unsigned* status = nullptr;
  void* dispatch_scratch = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
OncePerDevice<kMaxDevices> g_dev_once;

// Per-device set-up, done on the first call made with that device current.
DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceInfo& d = g_dev[dev];
  const cudaError_t e = g_dev_once.run(dev, [&]() -> cudaError_t {
    cudaError_t r = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (r != cudaSuccess) return r;
    void* p = nullptr;
    if ((r = cudaGetSymbolAddress(&p, g_status_word)) != cudaSuccess) return r;
    d.status = static_cast<unsigned*>(p);
    if ((r = cudaGetSymbolAddress(&p, g_dispatch_scratch)) != cudaSuccess) return r;
    d.dispatch_scratch = p;
    return cudaSuccess;
  });
  return e == cudaSuccess ? &d : nullptr;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline size_t act_bytes(const moe_config* c) { return c->act_dtype == MOE_BF16 ? 2 : 4; }

moe_status check_cfg(const moe_config* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d <= 0 || c->E <= 0 || c->E > 256 || c->k < 1 || c->k > c->E || c->k > 32 ||
      c->H <= 0 || c->n_shared < 0 || (c->n_shared > 0 && c->H_shared <= 0))
    return MOE_ERR_INVALID_ARG;
  if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->gating < MOE_GATE_SOFTMAX_TOPK || c->gating > MOE_GATE_SIGMOID_TOPK)
    return MOE_ERR_INVALID_ARG;
  if (c->residual < MOE_RES_NONE || c->residual > MOE_RES_INPUT_PLUS_EXTERNAL)
    return MOE_ERR_INVALID_ARG;
  // At most 2^24 routed pairs per call: the grouped GEMM packs an expert's 256-row pair
  // count into 16 bits, so no expert may hold 2^24 rows or more.
  if (static_cast<long long>(c->T) * c->k > (1ll << 24)) return MOE_ERR_UNSUPPORTED;
  if (c->act_dtype == MOE_BF16) {
    if (c->d % 256 || c->H % 128 || (c->n_shared > 0 && c->H_shared % 128))
      return MOE_ERR_UNSUPPORTED;
  } else {
    if (c->d % 64 || c->H % 64 || (c->n_shared > 0 && c->H_shared % 64)) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

#define MOE_REQUIRE(cond, code) \
  do {                          \
    if (!(cond)) return (code); \
  } while (0)
#define MOE_PTR(p) MOE_REQUIRE((p) != nullptr && aligned16(p), MOE_ERR_INVALID_ARG)
#define MOE_OPT_PTR(p) MOE_REQUIRE((p) == nullptr || aligned16(p), MOE_ERR_INVALID_ARG)
#define MOE_CUDA(expr)                                   \
  do {                                                   \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA;      \
  } while (0)

// Bump allocator over a caller workspace.
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = align256(off + count * sizeof(T));
    return p;
  }
};

// ------------------------------------------------------------------ expert FFN scratch
struct FfnScratch {
  int4* mt_routed;
  int32_t* gmb_routed;
  int4* mt_shared;
  int32_t* gmb_shared;
  void* h;
  void* h_shared;
  int32_t* rep_rows;   // compact list of the representatives' slots
  int32_t* rep_local;  // the same per bucket, at the bucket's own slots
  int32_t* rep_counts;
  int32_t* rep_off;
  void* x_rep;
};

size_t carve_ffn(const moe_config* c, bool condense, void* ws, FfnScratch* s) {
  const long long P = static_cast<long long>(c->T) * c->k;
  const size_t ab = act_bytes(c);
  Carver cv(ws);
  FfnScratch t;
  t.mt_routed = cv.take<int4>(max_mtiles(P, c->E));
  t.gmb_routed = cv.take<int32_t>(c->E + 1);
  t.mt_shared = cv.take<int4>(max_mtiles(c->T, 1));
  t.gmb_shared = cv.take<int32_t>(2);
  t.h = cv.take<char>(static_cast<size_t>(P) * c->H * ab);
  t.h_shared = cv.take<char>(static_cast<size_t>(c->T) * c->n_shared * c->H_shared * ab);
  t.rep_rows = t.rep_local = t.rep_counts = t.rep_off = nullptr;
  t.x_rep = nullptr;
  if (condense) {
    t.rep_rows = cv.take<int32_t>(P);
    t.rep_local = cv.take<int32_t>(P);
    t.rep_counts = cv.take<int32_t>(c->E);
    t.rep_off = cv.take<int32_t>(c->E + 1);
    t.x_rep = cv.take<char>(static_cast<size_t>(P) * c->d * ab);
  }
  if (s) *s = t;
  return cv.off;
}

// Routed experts: m-tile tables, gate/up + SwiGLU, down projection.
moe_status run_routed_ffn(const moe_config* c, const moe_weights* w, const void* x_perm,
                          const int32_t* offsets, const int32_t* rep_of, void* y_perm,
                          const FfnScratch& s, DeviceInfo* di, cudaStream_t st) {
  const int T = c->T, d = c->d, E = c->E, H = c->H;
  const long long P = static_cast<long long>(T) * c->k;
  // Rows the routed experts run on: every slot, or the representatives only.
  const void* A1 = x_perm;
  const int32_t* rowmap = nullptr;
  if (rep_of) {
    MOE_CUDA(launch_compact_reps(rep_of, offsets, E, s.rep_local, s.rep_counts, st));
    MOE_CUDA(launch_build_mtiles(s.rep_counts, nullptr, 0, E, s.rep_off, s.mt_routed,
                                 s.gmb_routed, st));
    MOE_CUDA(launch_gather_reps(c->act_dtype, x_perm, s.rep_local, offsets, s.rep_off, E,
                                static_cast<int>(P), d, s.x_rep, s.rep_rows, st));
    A1 = s.x_rep;
    rowmap = s.rep_rows;
  } else if (c->act_dtype != MOE_BF16) {
    MOE_CUDA(launch_build_mtiles(nullptr, offsets, 0, E, nullptr, s.mt_routed, s.gmb_routed, st));
  }
  if (c->act_dtype == MOE_BF16) {
    TcGemmArgs a = {};
    a.status = di->status;
    // gate/up + SwiGLU; the pair kernel reads the buckets' rows from the offsets (all slots)
    // or from the representatives' m-tile table
    a.mt_info = s.mt_routed;
    a.group_mt_begin = s.gmb_routed;
    a.group_off = rep_of ? nullptr : offsets;
    a.n_groups = E;
    // a bucket holds each token at most once: with at most 128 tokens every group is a tail
    a.tails_only = T <= 2 * kTailOnlyRows ? 1 : 0;
    a.n_ntiles = H / 128;
    a.nt_per_slice = H / 128;
    a.n_kblocks = d / kTcTileK;
    a.kb_per_slice = a.n_kblocks;
    a.b_up_offset = H;
    a.out = static_cast<__nv_bfloat16*>(s.h);
    a.ld_out = H;
    MOE_CUDA(tc_gemm(kTcSwiGLU, A1, P, d, w->W_gu, E, 2 * H, d, a, di->num_sms, st));
    // down projection
    a.n_ntiles = d / kTcTileN;
    a.nt_per_slice = a.n_ntiles;
    a.n_kblocks = H / kTcTileK;
    a.kb_per_slice = a.n_kblocks;
    a.b_up_offset = 0;
    a.out = static_cast<__nv_bfloat16*>(y_perm);
    a.ld_out = d;
    a.out_rowmap = rowmap;
    MOE_CUDA(tc_gemm(kTcStore, s.h, P, H, w->W_down, E, d, H, a, di->num_sms, st));
  } else {
    const int mt_max = max_mtiles(P, E);
    MOE_CUDA(simt_gemm_swiglu(static_cast<const float*>(A1), static_cast<const float*>(w->W_gu), E,
                              2 * H, d, 0, H / 64, H, H, s.mt_routed, s.gmb_routed, E, mt_max,
                              static_cast<float*>(s.h), st));
    MOE_CUDA(simt_gemm_store(static_cast<const float*>(s.h), static_cast<const float*>(w->W_down),
                             E, d, H, H, d, s.mt_routed, s.gmb_routed, E, mt_max, rowmap,
                             static_cast<float*>(y_perm), st));
  }
  return MOE_OK;
}

// Shared experts on all T rows of x: shared_out[t] = sum over shared experts.
// Uses only its own scratch (mt_shared, gmb_shared, h_shared), so it may run
// on another stream concurrently with run_routed_ffn.
moe_status run_shared_ffn(const moe_config* c, const moe_weights* w, const void* x,
                          void* shared_out, const FfnScratch& s, DeviceInfo* di, cudaStream_t st) {
  const int T = c->T, d = c->d, S = c->n_shared, Hs = c->H_shared;
  if (S == 0) return MOE_OK;
  if (c->act_dtype != MOE_BF16)
    MOE_CUDA(launch_build_mtiles(nullptr, nullptr, T, 1, nullptr, s.mt_shared, s.gmb_shared, st));
  if (c->act_dtype == MOE_BF16) {
    TcGemmArgs b = {};
    b.status = di->status;
    b.fixed_rows = T;  // one group of all T tokens
    b.n_groups = 1;
    b.tails_only = T <= 2 * kTailOnlyRows ? 1 : 0;
    b.n_ntiles = S * Hs / 128;
    b.nt_per_slice = Hs / 128;
    b.n_kblocks = d / kTcTileK;
    b.kb_per_slice = b.n_kblocks;
    b.b_up_offset = Hs;
    b.out = static_cast<__nv_bfloat16*>(s.h_shared);
    b.ld_out = static_cast<long long>(S) * Hs;
    MOE_CUDA(tc_gemm(kTcSwiGLU, x, T, d, w->Ws_gu, S, 2 * Hs, d, b, di->num_sms, st));
    b.n_ntiles = d / kTcTileN;
    b.nt_per_slice = b.n_ntiles;
    b.n_kblocks = S * Hs / kTcTileK;
    b.kb_per_slice = Hs / kTcTileK;
    b.b_up_offset = 0;
    b.out = static_cast<__nv_bfloat16*>(shared_out);
    b.ld_out = d;
    MOE_CUDA(tc_gemm(kTcStore, s.h_shared, T, S * Hs, w->Ws_down, S, d, Hs, b, di->num_sms, st));
  } else {
    const int mt_max = max_mtiles(T, 1);
    MOE_CUDA(simt_gemm_swiglu(static_cast<const float*>(x), static_cast<const float*>(w->Ws_gu), S,
                              2 * Hs, d, 0, Hs / 64, S * Hs, Hs, s.mt_shared, s.gmb_shared, 1,
                              mt_max, static_cast<float*>(s.h_shared), st));
    MOE_CUDA(simt_gemm_store(static_cast<const float*>(s.h_shared),
                             static_cast<const float*>(w->Ws_down), S, d, S * Hs, Hs, d,
                             s.mt_shared, s.gmb_shared, 1, mt_max, nullptr,
                             static_cast<float*>(shared_out), st));
  }
  return MOE_OK;
}

moe_status run_expert_ffn(const moe_config* c, const moe_weights* w, const void* x_perm,
                          const int32_t* offsets, const int32_t* rep_of, const void* x,
                          void* y_perm, void* shared_out, const FfnScratch& s, DeviceInfo* di,
                          cudaStream_t st) {
  if (c->T == 0) return MOE_OK;
  moe_status r = run_routed_ffn(c, w, x_perm, offsets, rep_of, y_perm, s, di, st);
  if (r != MOE_OK) return r;
  return run_shared_ffn(c, w, x, shared_out, s, di, st);
}

moe_status check_weights(const moe_config* c, const moe_weights* w) {
  MOE_REQUIRE(w != nullptr, MOE_ERR_INVALID_ARG);
  MOE_PTR(w->W_gu);
  MOE_PTR(w->W_down);
  if (c->n_shared > 0) {
    MOE_PTR(w->Ws_gu);
    MOE_PTR(w->Ws_down);
  }
  return MOE_OK;
}

// ------------------------------------------------------------------ router
// Workspace sizes must be computable without a device, so they assume the
// largest SM count the split-K choice can see; launches clamp to it as well.
constexpr int kMaxSmsForSizing = 256;

size_t route_ws_bytes(const moe_config* c) {
  if (c->act_dtype != MOE_BF16 || c->T == 0) return 0;
  return router_scratch_bytes(c->T, c->d, c->E, kMaxSmsForSizing);
}

moe_status run_router(const moe_config* c, const void* x, const float* W_r, const float* bias,
                      float* logits, int32_t* idx, float* gate, void* ws, DeviceInfo* di,
                      cudaStream_t st) {
  if (c->act_dtype == MOE_BF16) {
    const float* part = nullptr;
    int n_split = 0, ld = 0;
    MOE_CUDA(launch_router_tc(x, W_r, c->T, c->d, c->E,
                              di->num_sms < kMaxSmsForSizing ? di->num_sms : kMaxSmsForSizing,
                              ws, &part, &n_split, &ld, di->status, st));
    MOE_CUDA(launch_router_topk(part, n_split, ld, bias, logits, idx, gate, c->T, c->E, c->k,
                                c->gating, st));
  } else {
    MOE_CUDA(launch_router_logits(c->act_dtype, x, W_r, bias, logits, c->T, c->d, c->E, st));
    MOE_CUDA(launch_router_topk(logits, 1, c->E, nullptr, nullptr, idx, gate, c->T, c->E, c->k,
                                c->gating, st));
  }
  return MOE_OK;
}

// ------------------------------------------------------------------ layer workspace
struct LayerScratch {
  float* logits;
  void* route_ws;
  int32_t* topk_idx;
  float* gate;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* slot_of;
  void* x_perm;
  void* dispatch_ws;
  int32_t* rep_of;
  int32_t* n_rep;
  int32_t* n_condensed;
  void* condense_ws;
  void* y_perm;
  void* shared_out;
  void* ffn_ws;
};

size_t carve_layer(const moe_config* c, bool condense, void* ws, LayerScratch* s) {
  const long long P = static_cast<long long>(c->T) * c->k;
  const size_t ab = act_bytes(c);
  Carver cv(ws);
  LayerScratch t;
  t.logits = cv.take<float>(static_cast<size_t>(c->T) * c->E);
  t.route_ws = cv.take<char>(route_ws_bytes(c));
  t.topk_idx = cv.take<int32_t>(P);
  t.gate = cv.take<float>(P);
  t.counts = cv.take<int32_t>(c->E);
  t.offsets = cv.take<int32_t>(c->E + 1);
  t.perm = cv.take<int32_t>(P);
  t.slot_of = cv.take<int32_t>(P);
  t.x_perm = cv.take<char>(static_cast<size_t>(P) * c->d * ab);
  t.dispatch_ws = cv.take<char>(dispatch_auto_scratch_bytes(c->T, c->k, c->E) +
                                dispatch_scratch_bytes(c->T, c->E));
  t.rep_of = cv.take<int32_t>(P);
  t.n_rep = cv.take<int32_t>(c->E);
  t.n_condensed = cv.take<int32_t>(1);
  t.condense_ws = condense ? cv.take<char>(condense_scratch_bytes(c->T, c->k, c->E)) : nullptr;
  t.y_perm = cv.take<char>(static_cast<size_t>(P) * c->d * ab);
  t.shared_out = cv.take<char>(c->n_shared > 0 ? static_cast<size_t>(c->T) * c->d * ab : 0);
  t.ffn_ws = cv.take<char>(carve_ffn(c, condense, nullptr, nullptr));
  if (s) *s = t;
  return cv.off;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE_INDEX: return "device index out of range";
  }
  return "unknown status";
}

float moe_adaptive_tau(float l_norm) {
  return static_cast<float>(1.0 / (1.0 + exp(static_cast<double>(l_norm))));
}

moe_status moe_get_device_status(moe_stream_t stream) {
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned v = 0;
  MOE_CUDA(cudaStreamSynchronize(st));
  MOE_CUDA(cudaMemcpyAsync(&v, di->status, sizeof(v), cudaMemcpyDeviceToHost, st));
  MOE_CUDA(cudaMemsetAsync(di->status, 0, sizeof(unsigned), st));
  MOE_CUDA(cudaStreamSynchronize(st));
  return static_cast<moe_status>(v);
}

size_t moe_route_workspace_size(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return route_ws_bytes(cfg);
}

moe_status moe_route(const moe_config* cfg, const void* x, const float* W_r, const float* bias,
                     float* logits, int32_t* topk_idx, float* topk_gate, void* ws, size_t ws_bytes,
                     moe_stream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  MOE_PTR(x);
  MOE_PTR(W_r);
  MOE_OPT_PTR(bias);
  MOE_PTR(logits);
  MOE_PTR(topk_idx);
  MOE_PTR(topk_gate);
  const size_t need = route_ws_bytes(cfg);
  if (need > 0) MOE_PTR(ws);
  MOE_REQUIRE(ws_bytes >= need, MOE_ERR_WORKSPACE);
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  return run_router(cfg, x, W_r, bias, logits, topk_idx, topk_gate, ws, di,
                    reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_dispatch_workspace_size(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  const size_t a = dispatch_scratch_bytes(cfg->T, cfg->E);
  const size_t b = dispatch_auto_scratch_bytes(cfg->T, cfg->k, cfg->E);
  return align256(a > b ? a : b);
}

moe_status moe_dispatch(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                        int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* slot_of,
                        void* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  MOE_PTR(counts);
  MOE_PTR(offsets);
  if (cfg->T > 0) {
    MOE_PTR(x);
    MOE_PTR(topk_idx);
    MOE_PTR(perm);
    MOE_PTR(slot_of);
    MOE_PTR(x_perm);
  }
  MOE_OPT_PTR(ws);
  MOE_REQUIRE(ws_bytes >= moe_dispatch_workspace_size(cfg), MOE_ERR_WORKSPACE);
  MOE_REQUIRE(ws != nullptr || moe_dispatch_workspace_size(cfg) == 0, MOE_ERR_WORKSPACE);
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  MOE_CUDA(launch_dispatch_auto(cfg->act_dtype, x, topk_idx, cfg->T, cfg->d, cfg->E, cfg->k,
                                counts, offsets, perm, slot_of, x_perm, ws, di->num_sms,
                                di->status, st));
  return MOE_OK;
}

size_t moe_condense_workspace_size(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return align256(condense_scratch_bytes(cfg->T, cfg->k, cfg->E));
}

moe_status moe_condense(const moe_config* cfg, const void* x_perm, const int32_t* offsets, float tau,
                        int32_t* rep_of, int32_t* n_rep, int32_t* n_condensed, void* ws,
                        size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  MOE_PTR(offsets);
  MOE_PTR(n_rep);
  MOE_PTR(n_condensed);
  const long long P = static_cast<long long>(cfg->T) * cfg->k;
  if (P > 0) {
    MOE_PTR(x_perm);
    MOE_PTR(rep_of);
  }
  const bool active = tau <= 1.0f;
  if (active) {
    if (cfg->act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (cfg->T > kCondenseMaxTokens) return MOE_ERR_UNSUPPORTED;
    MOE_PTR(ws);
    MOE_REQUIRE(ws_bytes >= moe_condense_workspace_size(cfg), MOE_ERR_WORKSPACE);
  }
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  MOE_CUDA(launch_condense(static_cast<const __nv_bfloat16*>(x_perm), offsets, cfg->T, cfg->k,
                           cfg->d, cfg->E, tau, di->num_sms, rep_of, n_rep, n_condensed, ws,
                           di->status, st));
  return MOE_OK;
}

size_t moe_condense_history_bytes(const moe_config* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return hist_record_bytes(cfg->T, cfg->k, cfg->E);
}

moe_status moe_condense_hist(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                             const int32_t* perm, const int32_t* slot_of, float tau, float s1,
                             float s2, const void* hist_in, void* hist_out, int32_t* rep_of,
                             int32_t* n_rep, int32_t* n_condensed, int32_t* n_cos_tiles,
                             void* ws, size_t ws_bytes, moe_stream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (!(tau <= 1.0f) || s1 != s1 || s2 != s2) return MOE_ERR_INVALID_ARG;
  if (cfg->act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  const long long P = static_cast<long long>(cfg->T) * cfg->k;
  if (cfg->T > kCondenseMaxTokens) return MOE_ERR_UNSUPPORTED;
  MOE_PTR(offsets);
  MOE_PTR(n_rep);
  MOE_PTR(n_condensed);
  MOE_OPT_PTR(n_cos_tiles);
  MOE_OPT_PTR(hist_in);
  MOE_PTR(hist_out);
  if (P > 0) {
    MOE_PTR(x_perm);
    MOE_PTR(rep_of);
    MOE_PTR(perm);
    MOE_PTR(slot_of);
  }
  const size_t rec = hist_record_bytes(cfg->T, cfg->k, cfg->E);
  if (hist_in) {
    const char* a = static_cast<const char*>(hist_in);
    const char* b = static_cast<const char*>(hist_out);
    MOE_REQUIRE(a + rec <= b || b + rec <= a, MOE_ERR_INVALID_ARG);
  }
  MOE_PTR(ws);
  MOE_REQUIRE(ws_bytes >= moe_condense_workspace_size(cfg), MOE_ERR_WORKSPACE);
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  HistArgs h;
  h.perm = perm;
  h.slot_of = slot_of;
  h.T = cfg->T;
  h.k = cfg->k;
  h.s1 = s1;
  h.s2 = s2;
  h.hist_in = hist_in;
  h.hist_out = hist_out;
  h.n_cos_tiles = n_cos_tiles;
  MOE_CUDA(launch_condense_hist(static_cast<const __nv_bfloat16*>(x_perm), offsets,
                                cfg->d, cfg->E, tau, h, di->num_sms, rep_of,
                                n_rep, n_condensed, ws, di->status,
                                reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

size_t moe_expert_ffn_workspace_size(const moe_config* cfg, int with_condensation) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return carve_ffn(cfg, with_condensation != 0, nullptr, nullptr);
}

moe_status moe_expert_ffn(const moe_config* cfg, const moe_weights* w, const void* x_perm,
                          const int32_t* offsets, const int32_t* rep_of, const void* x,
                          void* y_perm, void* shared_out, void* ws, size_t ws_bytes,
                          moe_stream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  s = check_weights(cfg, w);
  if (s != MOE_OK) return s;
  MOE_PTR(x_perm);
  MOE_PTR(offsets);
  MOE_OPT_PTR(rep_of);
  MOE_PTR(y_perm);
  if (cfg->n_shared > 0) {
    MOE_PTR(x);
    MOE_PTR(shared_out);
  }
  MOE_PTR(ws);
  MOE_REQUIRE(ws_bytes >= moe_expert_ffn_workspace_size(cfg, rep_of != nullptr), MOE_ERR_WORKSPACE);
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  FfnScratch fs;
  carve_ffn(cfg, rep_of != nullptr, ws, &fs);
  return run_expert_ffn(cfg, w, x_perm, offsets, rep_of, x, y_perm, shared_out, fs, di,
                        reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_combine(const moe_config* cfg, const void* y_perm, const void* shared_out,
                       const int32_t* slot_of, const int32_t* rep_of, const float* topk_gate,
                       const void* x, const void* residual, void* out, moe_stream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  MOE_PTR(y_perm);
  MOE_OPT_PTR(shared_out);
  MOE_REQUIRE(cfg->n_shared == 0 || shared_out != nullptr, MOE_ERR_INVALID_ARG);
  MOE_PTR(slot_of);
  MOE_OPT_PTR(rep_of);
  MOE_PTR(topk_gate);
  MOE_PTR(out);
  if (cfg->residual == MOE_RES_INPUT || cfg->residual == MOE_RES_INPUT_PLUS_EXTERNAL) MOE_PTR(x);
  if (cfg->residual == MOE_RES_EXTERNAL || cfg->residual == MOE_RES_INPUT_PLUS_EXTERNAL)
    MOE_PTR(residual);
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  MOE_CUDA(launch_combine(cfg->act_dtype, y_perm, cfg->n_shared > 0 ? shared_out : nullptr, slot_of,
                          rep_of, topk_gate, x, residual, cfg->residual, out, cfg->T, cfg->d,
                          cfg->k, cfg->T * cfg->k, di->status,
                          reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}

size_t moe_workspace_size(const moe_config* cfg, int with_condensation) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return carve_layer(cfg, with_condensation != 0, nullptr, nullptr);
}

}  // extern "C"

namespace moe {
namespace {

// Fork/join events of moe_layer_forward_ex, one pair per host thread and device
// (created on first use, kept for the life of the process), so concurrent
// callers on different threads never share one.
thread_local cudaEvent_t t_events[kMaxDevices][2] = {};

bool overlap_events(cudaEvent_t** ev) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  for (int i = 0; i < 2; ++i)
    if (!t_events[dev][i] &&
        cudaEventCreateWithFlags(&t_events[dev][i], cudaEventDisableTiming) != cudaSuccess)
      return false;
  *ev = t_events[dev];
  return true;
}

moe_status layer_forward_impl(const moe_config* cfg, const moe_weights* w, const void* x,
                              const void* residual, float tau, void* out, void* partial_out,
                              int32_t* topk_idx_out, int32_t* n_condensed_out, void* ws,
                              size_t ws_bytes, cudaStream_t st, cudaStream_t aux) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  s = check_weights(cfg, w);
  if (s != MOE_OK) return s;
  MOE_PTR(w->W_r);
  MOE_OPT_PTR(w->router_bias);
  MOE_PTR(x);
  MOE_PTR(out);
  MOE_OPT_PTR(partial_out);
  MOE_OPT_PTR(topk_idx_out);
  MOE_OPT_PTR(n_condensed_out);
  if (cfg->residual == MOE_RES_EXTERNAL || cfg->residual == MOE_RES_INPUT_PLUS_EXTERNAL)
    MOE_PTR(residual);
  const bool condense = tau <= 1.0f;
  const long long P = static_cast<long long>(cfg->T) * cfg->k;
  if (condense && (cfg->act_dtype != MOE_BF16 || cfg->T > kCondenseMaxTokens))
    return MOE_ERR_UNSUPPORTED;
  MOE_PTR(ws);
  MOE_REQUIRE(ws_bytes >= moe_workspace_size(cfg, condense), MOE_ERR_WORKSPACE);
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  LayerScratch L;
  carve_layer(cfg, condense, ws, &L);
  FfnScratch fs;
  carve_ffn(cfg, condense, L.ffn_ws, &fs);
  const bool overlap = aux != nullptr && aux != st && cfg->n_shared > 0;
  cudaEvent_t* ev = nullptr;
  if (overlap && !overlap_events(&ev)) return MOE_ERR_CUDA;

  int32_t* idx = topk_idx_out ? topk_idx_out : L.topk_idx;
  s = run_router(cfg, x, w->W_r, w->router_bias, L.logits, idx, L.gate, L.route_ws, di, st);
  if (s != MOE_OK) return s;
  if (overlap) {
    // The shared experts need only x: they start on the second stream once the
    // router is done (the router's tensor-core GEMM would not fit beside them
    // on an SM) and run beside dispatch and the routed experts.
    MOE_CUDA(cudaEventRecord(ev[0], st));
    MOE_CUDA(cudaStreamWaitEvent(aux, ev[0], 0));
    s = run_shared_ffn(cfg, w, x, L.shared_out, fs, di, aux);
    if (s != MOE_OK) return s;
    MOE_CUDA(cudaEventRecord(ev[1], aux));
  }
  // a condensing layer has the dispatch form the slots' row norms and hashes as it moves the
  // rows, where the condensation reads them
  const bool stats = condense && cfg->T * cfg->k > 0;
  RowStatsOut rs = {};
  if (stats) rs = condense_stats_ptrs(L.condense_ws, cfg->T, cfg->k, cfg->E);
  MOE_CUDA(launch_dispatch_auto(cfg->act_dtype, x, idx, cfg->T, cfg->d, cfg->E, cfg->k,
                                L.counts, L.offsets, L.perm, L.slot_of, L.x_perm, L.dispatch_ws,
                                di->num_sms, di->status, st, stats ? &rs : nullptr));
  const int32_t* rep_of = nullptr;
  if (condense) {
    MOE_CUDA(launch_condense(static_cast<const __nv_bfloat16*>(L.x_perm), L.offsets,
                             cfg->T, cfg->k, cfg->d, cfg->E, tau, di->num_sms, L.rep_of,
                             L.n_rep, n_condensed_out ? n_condensed_out : L.n_condensed,
                             L.condense_ws, di->status, st, stats));
    rep_of = L.rep_of;
  } else if (n_condensed_out) {
    MOE_CUDA(cudaMemsetAsync(n_condensed_out, 0, sizeof(int32_t), st));
  }
  s = run_routed_ffn(cfg, w, L.x_perm, L.offsets, rep_of, L.y_perm, fs, di, st);
  if (s != MOE_OK) return s;
  if (overlap) {
    MOE_CUDA(cudaStreamWaitEvent(st, ev[1], 0));
  } else {
    s = run_shared_ffn(cfg, w, x, L.shared_out, fs, di, st);
    if (s != MOE_OK) return s;
  }
  // The kernel before the combine (a down-projection GEMM) triggers its dependents only
  // after its own wait, and the router waited for the caller's work before reading x, so
  // x and residual are complete whenever the combine starts.
  MOE_CUDA(launch_combine(cfg->act_dtype, L.y_perm, cfg->n_shared > 0 ? L.shared_out : nullptr,
                          L.slot_of, rep_of, L.gate, x, residual, cfg->residual, out, cfg->T,
                          cfg->d, cfg->k, static_cast<int>(P), di->status, st, partial_out,
                          /*inputs_ready=*/true));
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const void* x,
                             const void* residual, float tau, void* out, int32_t* topk_idx_out,
                             int32_t* n_condensed_out, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
  return moe::layer_forward_impl(cfg, w, x, residual, tau, out, nullptr, topk_idx_out,
                                 n_condensed_out, ws, ws_bytes,
                                 reinterpret_cast<cudaStream_t>(stream), nullptr);
}

moe_status moe_layer_forward_ex(const moe_config* cfg, const moe_weights* w, const void* x,
                                const void* residual, float tau, void* out, void* partial_out,
                                int32_t* topk_idx_out, int32_t* n_condensed_out, void* ws,
                                size_t ws_bytes, moe_stream_t stream, moe_stream_t aux_stream) {
  return moe::layer_forward_impl(cfg, w, x, residual, tau, out, partial_out, topk_idx_out,
                                 n_condensed_out, ws, ws_bytes,
                                 reinterpret_cast<cudaStream_t>(stream),
                                 reinterpret_cast<cudaStream_t>(aux_stream));
}

}  // extern "C"

// ------------------------------------------------------------------ layer backward
namespace moe {
namespace {

struct BwdScratch {
  float* logits;
  void* route_ws;
  int32_t* idx;
  float* gate;
  int32_t* counts;
  int32_t* offsets;
  int32_t* perm;
  int32_t* slot_of;
  void* x_perm;
  void* dispatch_ws;
  int32_t* pcounts;
  int32_t* poffsets;
  int4* mt;
  int32_t* gmb;
  void* x_pad;
  void* au;
  void* h;
  void* y;
  void* dy;
  void* dA;
  float* dz;
  float* dg;
  float* dl;
  float* dx_router;
  void* router_ws;
  // shared experts
  void* x_s;
  void* dout_s;
  void* au_s;
  void* h_s;
  void* dA_s;
  float* dz_s;
  int4* mt_s;
  int32_t* gmb_s;
  // condensation
  void* condense_ws;
  int32_t* rep_of;
  int32_t* n_rep;
  int32_t* n_condensed;
  int32_t* mem_off;
  int32_t* mem_cnt;
  int32_t* mem_list;
};

// rows of the padded slot space: every group rounded up to kBwdPad rows
long long bwd_rows_max(const moe_config* c) {
  return static_cast<long long>(c->T) * c->k + static_cast<long long>(kBwdPad) * c->E;
}
int bwd_tokens_padded(const moe_config* c) { return (c->T + kBwdPad - 1) / kBwdPad * kBwdPad; }

size_t carve_bwd(const moe_config* c, bool condense, void* ws, BwdScratch* s) {
  const long long P = static_cast<long long>(c->T) * c->k;
  const long long R = bwd_rows_max(c);
  const int Tp = bwd_tokens_padded(c);
  const size_t d = c->d, H = c->H, S = c->n_shared, Hs = c->H_shared;
  Carver cv(ws);
  BwdScratch t;
  t.logits = cv.take<float>(static_cast<size_t>(c->T) * c->E);
  t.route_ws = cv.take<char>(route_ws_bytes(c));
  t.idx = cv.take<int32_t>(P);
  t.gate = cv.take<float>(P);
  t.counts = cv.take<int32_t>(c->E);
  t.offsets = cv.take<int32_t>(c->E + 1);
  t.perm = cv.take<int32_t>(P);
  t.slot_of = cv.take<int32_t>(P);
  t.x_perm = cv.take<__nv_bfloat16>(P * d);
  t.dispatch_ws = cv.take<char>(dispatch_auto_scratch_bytes(c->T, c->k, c->E));
  t.pcounts = cv.take<int32_t>(c->E);
  t.poffsets = cv.take<int32_t>(c->E + 1);
  t.mt = cv.take<int4>(max_mtiles(R, c->E));
  t.gmb = cv.take<int32_t>(c->E + 1);
  t.x_pad = cv.take<__nv_bfloat16>(R * d);
  t.au = cv.take<__nv_bfloat16>(R * 2 * H);
  t.h = cv.take<__nv_bfloat16>(R * H);
  t.y = cv.take<__nv_bfloat16>(R * d);
  t.dy = cv.take<__nv_bfloat16>(R * d);
  t.dA = cv.take<__nv_bfloat16>(R * 2 * H);
  t.dz = cv.take<float>(R * d);
  t.dg = cv.take<float>(P);
  t.dl = cv.take<float>(static_cast<size_t>(c->T) * c->E);
  t.dx_router = cv.take<float>(static_cast<size_t>(c->T) * d);
  t.router_ws = cv.take<char>(router_bwd_scratch_bytes(c->T, c->d, c->E));
  t.x_s = t.dout_s = t.au_s = t.h_s = t.dA_s = nullptr;
  t.dz_s = nullptr;
  t.mt_s = nullptr;
  t.gmb_s = nullptr;
  if (S > 0) {
    t.x_s = cv.take<__nv_bfloat16>(Tp * d);
    t.dout_s = cv.take<__nv_bfloat16>(Tp * d);
    t.au_s = cv.take<__nv_bfloat16>(Tp * S * 2 * Hs);
    t.h_s = cv.take<__nv_bfloat16>(Tp * S * Hs);
    t.dA_s = cv.take<__nv_bfloat16>(Tp * S * 2 * Hs);
    t.dz_s = cv.take<float>(Tp * d);
    t.mt_s = cv.take<int4>(max_mtiles(Tp, 1));
    t.gmb_s = cv.take<int32_t>(2);
  }
  t.condense_ws = nullptr;
  t.rep_of = t.n_rep = t.n_condensed = t.mem_off = t.mem_cnt = t.mem_list = nullptr;
  if (condense) {
    t.condense_ws = cv.take<char>(condense_scratch_bytes(c->T, c->k, c->E));
    t.rep_of = cv.take<int32_t>(P);
    t.n_rep = cv.take<int32_t>(c->E);
    t.n_condensed = cv.take<int32_t>(1);
    t.mem_off = cv.take<int32_t>(P);
    t.mem_cnt = cv.take<int32_t>(P);
    t.mem_list = cv.take<int32_t>(P);
  }
  if (s) *s = t;
  return cv.off;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_layer_backward_workspace_size(const moe_config* cfg, int with_condensation) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return carve_bwd(cfg, with_condensation != 0, nullptr, nullptr);
}

extern "C" moe_status moe_layer_backward(const moe_config* cfg, const moe_weights* w,
                                         const void* x, const void* d_out, float tau, void* d_x,
                                         void* d_residual, float* dW_r, float* d_bias,
                                         float* dW_gu, float* dW_down, float* dWs_gu,
                                         float* dWs_down, void* ws, size_t ws_bytes,
                                         moe_stream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  if (cfg->T == 0) return MOE_OK;
  if (cfg->act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  const bool condense = tau <= 1.0f;
  if (condense && cfg->T > kCondenseMaxTokens) return MOE_ERR_UNSUPPORTED;
  s = check_weights(cfg, w);
  if (s != MOE_OK) return s;
  MOE_PTR(w->W_r);
  MOE_OPT_PTR(w->router_bias);
  MOE_PTR(x);
  MOE_PTR(d_out);
  MOE_PTR(d_x);
  MOE_OPT_PTR(d_residual);
  MOE_PTR(dW_r);
  MOE_OPT_PTR(d_bias);
  MOE_PTR(dW_gu);
  MOE_PTR(dW_down);
  if (cfg->n_shared > 0) {
    MOE_PTR(dWs_gu);
    MOE_PTR(dWs_down);
  }
  MOE_PTR(ws);
  MOE_REQUIRE(ws_bytes >= moe_layer_backward_workspace_size(cfg, condense), MOE_ERR_WORKSPACE);
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int T = cfg->T, d = cfg->d, E = cfg->E, k = cfg->k, H = cfg->H, S = cfg->n_shared,
            Hs = cfg->H_shared;
  const long long R = bwd_rows_max(cfg);
  const int Tp = bwd_tokens_padded(cfg);
  BwdScratch b;
  carve_bwd(cfg, condense, ws, &b);
  const int sms = di->num_sms;

  // forward recompute: routing, dispatch, padded slot space, [a | u], h, y
  s = run_router(cfg, x, w->W_r, w->router_bias, b.logits, b.idx, b.gate, b.route_ws, di, st);
  if (s != MOE_OK) return s;
  const bool stats = condense && T * k > 0;
  RowStatsOut rs = {};
  if (stats) rs = condense_stats_ptrs(b.condense_ws, T, k, E);
  MOE_CUDA(launch_dispatch_auto(cfg->act_dtype, x, b.idx, T, d, E, k, b.counts, b.offsets, b.perm,
                                b.slot_of, b.x_perm, b.dispatch_ws, sms, di->status, st,
                                stats ? &rs : nullptr));
  if (condense) {
    // Luffy condensation: a condensed slot's expert input is its representative's row
    MOE_CUDA(launch_condense(static_cast<const __nv_bfloat16*>(b.x_perm), b.offsets, T, k, d, E,
                             tau, sms, b.rep_of, b.n_rep, b.n_condensed, b.condense_ws, di->status,
                             st, stats));
    MOE_CUDA(launch_members(b.rep_of, b.offsets, E, b.mem_off, b.mem_cnt, b.mem_list, st));
  }
  MOE_CUDA(launch_pad_counts(b.counts, E, b.pcounts, st));
  MOE_CUDA(launch_build_mtiles(b.pcounts, nullptr, 0, E, b.poffsets, b.mt, b.gmb, st));
  MOE_CUDA(launch_pad_rows(b.x_perm, b.offsets, b.poffsets, b.rep_of, E, static_cast<int>(R), d,
                           b.x_pad, b.dy, st));
  {
    TcGemmArgs a = {};
    a.status = di->status;
    a.mt_info = b.mt;
    a.group_mt_begin = b.gmb;
    a.n_groups = E;
    a.n_ntiles = 2 * H / kTcTileN;
    a.nt_per_slice = a.n_ntiles;
    a.n_kblocks = d / kTcTileK;
    a.kb_per_slice = a.n_kblocks;
    a.out = static_cast<__nv_bfloat16*>(b.au);
    a.ld_out = 2 * H;
    MOE_CUDA(tc_gemm(kTcStore, b.x_pad, R, d, w->W_gu, E, 2 * H, d, a, sms, st));
  }
  MOE_CUDA(launch_swiglu_from_au(b.au, b.poffsets + E, static_cast<int>(R), 1, H, b.h, st));
  {
    TcGemmArgs a = {};
    a.status = di->status;
    a.mt_info = b.mt;
    a.group_mt_begin = b.gmb;
    a.n_groups = E;
    a.n_ntiles = d / kTcTileN;
    a.nt_per_slice = a.n_ntiles;
    a.n_kblocks = H / kTcTileK;
    a.kb_per_slice = a.n_kblocks;
    a.out = static_cast<__nv_bfloat16*>(b.y);
    a.ld_out = d;
    MOE_CUDA(tc_gemm(kTcStore, b.h, R, H, w->W_down, E, d, H, a, sms, st));
  }

  // combine and router backward
  MOE_CUDA(launch_combine_bwd(d_out, b.y, b.idx, b.slot_of, b.offsets, b.poffsets, b.gate, T, d,
                              k, b.dy, b.dg, st));
  MOE_CUDA(launch_router_bwd(b.logits, b.idx, b.gate, b.dg, T, E, k, cfg->gating, b.dl, st));
  MOE_CUDA(launch_router_param_grads(x, b.dl, w->W_r, T, d, E, dW_r,
                                     w->router_bias ? d_bias : nullptr, b.dx_router, b.router_ws,
                                     st));
  if (d_bias && !w->router_bias) MOE_CUDA(cudaMemsetAsync(d_bias, 0, sizeof(float) * E, st));

  // routed experts
  {
    BwdArgs a = {};
    a.status = di->status;
    a.mt_info = b.mt;
    a.group_mt_begin = b.gmb;
    a.n_groups = E;
    BwdGemmOperands op = {};
    // dA = SwiGLU'(dy . W_down)
    a.nt_per_slice = (H + 255) / 256;
    a.n_ntiles = a.nt_per_slice;
    a.n_kblocks = d / 64;
    a.n_per_slice = H;
    a.au = static_cast<const __nv_bfloat16*>(b.au);
    a.ld_au = 2 * H;
    a.out_bf16 = static_cast<__nv_bfloat16*>(b.dA);
    a.ld_out = 2 * H;
    op = {b.dy, d, R, w->W_down, H, d, E};
    MOE_CUDA(bwd_gemm(kBwdDH, op, a, sms, st));
    // dz = dA . W_gu
    a.n_ntiles = d / 256;
    a.n_kblocks = 2 * H / 64;
    a.kb_per_slice = a.n_kblocks;
    a.out_f32 = b.dz;
    a.ld_out = d;
    op = {b.dA, 2 * H, R, w->W_gu, d, 2 * H, E};
    MOE_CUDA(bwd_gemm(kBwdDX, op, a, sms, st));
    // dW_down[e] = dy^T . h
    a.n_mtiles = d / 256;
    a.n_ntiles = (H + 255) / 256;
    a.n_cols = H;
    a.group_rows = b.poffsets;
    a.out_f32 = dW_down;
    a.ld_out = H;
    a.out_group_stride = static_cast<long long>(d) * H;
    op = {b.dy, d, R, b.h, H, R, 1};
    MOE_CUDA(bwd_gemm(kBwdDWD, op, a, sms, st));
    // dW_gu[e] = dA^T . x
    a.n_mtiles = 2 * H / 256;
    a.n_ntiles = d / 256;
    a.out_f32 = dW_gu;
    a.ld_out = d;
    a.out_group_stride = 2ll * H * d;
    op = {b.dA, 2 * H, R, b.x_pad, d, R, 1};
    MOE_CUDA(bwd_gemm(kBwdDWGU, op, a, sms, st));
  }

  // shared experts: every token, gate 1, so their output gradient is d_out itself
  if (S > 0) {
    // x and d_out padded to Tp rows; when T is already a multiple of the pad they are used as is
    const void* xs = x;
    const void* douts = d_out;
    if (Tp != T) {
      MOE_CUDA(launch_pad_tokens(x, T, Tp, d, b.x_s, st));
      MOE_CUDA(launch_pad_tokens(d_out, T, Tp, d, b.dout_s, st));
      xs = b.x_s;
      douts = b.dout_s;
    }
    MOE_CUDA(launch_build_mtiles(nullptr, nullptr, Tp, 1, nullptr, b.mt_s, b.gmb_s, st));
    {
      TcGemmArgs a = {};
      a.status = di->status;
      a.mt_info = b.mt_s;
      a.group_mt_begin = b.gmb_s;
      a.n_groups = 1;
      a.n_ntiles = S * 2 * Hs / kTcTileN;
      a.nt_per_slice = 2 * Hs / kTcTileN;
      a.n_kblocks = d / kTcTileK;
      a.kb_per_slice = a.n_kblocks;
      a.out = static_cast<__nv_bfloat16*>(b.au_s);
      a.ld_out = static_cast<long long>(S) * 2 * Hs;
      MOE_CUDA(tc_gemm(kTcStore, xs, Tp, d, w->Ws_gu, S, 2 * Hs, d, a, sms, st));
    }
    MOE_CUDA(launch_swiglu_from_au(b.au_s, nullptr, Tp, S, Hs, b.h_s, st));
    BwdArgs a = {};
    a.status = di->status;
    a.mt_info = b.mt_s;
    a.group_mt_begin = b.gmb_s;
    a.n_groups = 1;
    BwdGemmOperands op = {};
    a.nt_per_slice = (Hs + 255) / 256;
    a.n_ntiles = S * a.nt_per_slice;
    a.n_kblocks = d / 64;
    a.n_per_slice = Hs;
    a.au = static_cast<const __nv_bfloat16*>(b.au_s);
    a.ld_au = static_cast<long long>(S) * 2 * Hs;
    a.out_bf16 = static_cast<__nv_bfloat16*>(b.dA_s);
    a.ld_out = a.ld_au;
    op = {douts, d, Tp, w->Ws_down, Hs, d, S};
    MOE_CUDA(bwd_gemm(kBwdDH, op, a, sms, st));
    a.n_ntiles = d / 256;
    a.n_kblocks = S * 2 * Hs / 64;
    a.kb_per_slice = 2 * Hs / 64;
    a.out_f32 = b.dz_s;
    a.ld_out = d;
    op = {b.dA_s, static_cast<long long>(S) * 2 * Hs, Tp, w->Ws_gu, d, 2 * Hs, S};
    MOE_CUDA(bwd_gemm(kBwdDX, op, a, sms, st));
    BwdArgs g = {};
    g.status = di->status;
    g.n_groups = S;
    g.group_rows = nullptr;
    g.rows_shared = Tp;
    g.n_mtiles = d / 256;
    g.n_ntiles = (Hs + 255) / 256;
    g.n_cols = Hs;
    g.b_col0 = 0;
    g.b_col_stride = Hs;
    g.out_f32 = dWs_down;
    g.ld_out = Hs;
    g.out_group_stride = static_cast<long long>(d) * Hs;
    op = {douts, d, Tp, b.h_s, static_cast<long long>(S) * Hs, Tp, 1};
    MOE_CUDA(bwd_gemm(kBwdDWD, op, g, sms, st));
    g.n_mtiles = 2 * Hs / 256;
    g.n_ntiles = d / 256;
    g.a_col_stride = 2 * Hs;
    g.out_f32 = dWs_gu;
    g.ld_out = d;
    g.out_group_stride = 2ll * Hs * d;
    op = {b.dA_s, static_cast<long long>(S) * 2 * Hs, Tp, xs, d, Tp, 1};
    MOE_CUDA(bwd_gemm(kBwdDWGU, op, g, sms, st));
  }

  // input gradient and the residual stream's gradient
  const bool dout_to_x =
      cfg->residual == MOE_RES_INPUT || cfg->residual == MOE_RES_INPUT_PLUS_EXTERNAL;
  MOE_CUDA(launch_dx_assemble(d_out, dout_to_x ? 1 : 0, b.dx_router, S > 0 ? b.dz_s : nullptr,
                              b.dz, b.idx, b.slot_of, b.offsets, b.poffsets, b.rep_of, b.mem_off,
                              b.mem_cnt, b.mem_list, T, d, k, d_x, st));
  if (d_residual) {
    if (cfg->residual == MOE_RES_EXTERNAL || cfg->residual == MOE_RES_INPUT_PLUS_EXTERNAL)
      MOE_CUDA(cudaMemcpyAsync(d_residual, d_out, static_cast<size_t>(T) * d * 2,
                               cudaMemcpyDeviceToDevice, st));
    else
      MOE_CUDA(cudaMemsetAsync(d_residual, 0, static_cast<size_t>(T) * d * 2, st));
  }
  return MOE_OK;
}

// ------------------------------------------------------------------ dispatch without a workspace
// For callers that cannot allocate device memory: the dispatch scratch lives
// in the file-scope device array g_dispatch_scratch instead of a caller workspace.
extern "C" moe_status moe_dispatch_static_scratch(const moe_config* cfg, const void* x,
                                                  const int32_t* topk_idx, int32_t* counts,
                                                  int32_t* offsets, int32_t* perm,
                                                  int32_t* slot_of, void* x_perm,
                                                  moe_stream_t stream) {
  moe_status s = check_cfg(cfg);
  if (s != MOE_OK) return s;
  MOE_PTR(counts);
  MOE_PTR(offsets);
  if (cfg->T > 0) {
    MOE_PTR(x);
    MOE_PTR(topk_idx);
    MOE_PTR(perm);
    MOE_PTR(slot_of);
    MOE_PTR(x_perm);
  }
  if (dispatch_scratch_bytes(cfg->T, cfg->E) > kStaticDispatchScratchBytes)
    return MOE_ERR_WORKSPACE;
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  MOE_CUDA(launch_dispatch(cfg->act_dtype, x, topk_idx, cfg->T, cfg->d, cfg->E, cfg->k, counts,
                           offsets, perm, slot_of, x_perm, di->dispatch_scratch,
                           di->status, reinterpret_cast<cudaStream_t>(stream)));
  return MOE_OK;
}
