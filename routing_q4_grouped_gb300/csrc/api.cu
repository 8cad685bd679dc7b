// api.cu — the extern "C" boundary of libmoeq4: argument validation,
// workspace layout, TMA descriptor encoding and the launch sequence.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moeq4.h"
#include "../../include/moeq4_debug.h"
#include "internal.h"

namespace moeq4 {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* base,
               uint64_t inner, uint64_t outer, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DevInfo {
  int sms = 0;
  bool sm103 = false;
};

// Per-device constants, looked up once per device.
moe_status device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> g(mu);
  if (!have[dev]) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    cache[dev].sms = sms;
    cache[dev].sm103 = (major == 10 && minor == 3);
    have[dev] = true;
  }
  *out = cache[dev];
  return out->sm103 ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

uint64_t timeout_ns() {
  static uint64_t t = [] {
    const char* s = std::getenv("MOEQ4_WAIT_TIMEOUT_MS");
    long ms = s ? std::atol(s) : 2000;
    if (ms <= 0) ms = 2000;
    return static_cast<uint64_t>(ms) * 1000000ull;
  }();
  return t;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_route_out(const moe_route_out* r) {
  if (!r) return MOE_ERR_ARG;
  if (r->T < 0 || r->E < 1 || r->E > 1024 || r->k < 1 || r->k > r->E || r->k > 32 ||
      r->block_m < 1 || r->block_m > 128)
    return MOE_ERR_ARG;
  if (static_cast<long long>(r->T) * r->k >= (1ll << 30)) return MOE_ERR_SHAPE;
  const void* always[] = {r->counts, r->offsets, r->tiles, r->n_tiles, r->err};
  const void* per_token[] = {r->ids, r->w, r->perm, r->inv};   // may be NULL when T == 0
  for (const void* p : always) {
    if (!p) return MOE_ERR_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  }
  for (const void* p : per_token) {
    if (!p && r->T > 0) return MOE_ERR_ARG;
    if (!aligned16(p)) return MOE_ERR_ALIGN;
  }
  return MOE_OK;
}

moe_status check_mat(const moe_q4_mat& m) {
  if (!m.qw || !m.scale || !m.bias) return MOE_ERR_ARG;
  if (!aligned16(m.qw) || !aligned16(m.scale) || !aligned16(m.bias)) return MOE_ERR_ALIGN;
  return MOE_OK;
}

moe_status check_dims(int E, int d, int f, int f_s) {
  if (E < 1 || E > 1024 || d < 1 || f < 1 || f_s < 0) return MOE_ERR_ARG;
  if (d % 256 || f % 128 || f_s % 128 || d > 16384 || f > 8192 || f_s > 8192) return MOE_ERR_SHAPE;
  return MOE_OK;
}

moe_status check_weights(const moe_q4_weights* W) {
  if (!W) return MOE_ERR_ARG;
  moe_status s = check_dims(W->E, W->d, W->f, W->f_s);
  if (s != MOE_OK) return s;
  if ((s = check_mat(W->gate_up)) != MOE_OK || (s = check_mat(W->down)) != MOE_OK) return s;
  if (W->f_s > 0 &&
      ((s = check_mat(W->sh_gate_up)) != MOE_OK || (s = check_mat(W->sh_down)) != MOE_OK))
    return s;
  return MOE_OK;
}

moe_status check_packed(const moe_q4_packed* W) {
  if (!W) return MOE_ERR_ARG;
  moe_status s = check_dims(W->E, W->d, W->f, W->f_s);
  if (s != MOE_OK) return s;
  if (!W->data) return MOE_ERR_ARG;
  if (!aligned16(W->data)) return MOE_ERR_ALIGN;
  return MOE_OK;
}

RouteArgs make_route_args(const float* logits, const moe_route_out* r, void* ws) {
  RouteArgs a{};
  const RouteWs L = route_ws_layout(r->T, r->E, r->k);
  char* base = static_cast<char*>(ws);
  a.logits = logits;
  a.T = r->T;
  a.E = r->E;
  a.k = r->k;
  a.block_m = r->block_m;
  a.ids = r->ids;
  a.w = r->w;
  a.counts = r->counts;
  a.offsets = r->offsets;
  a.perm = r->perm;
  a.inv = r->inv;
  a.tiles = r->tiles;
  a.n_tiles = r->n_tiles;
  a.err = r->err;
  a.rows = reinterpret_cast<uint32_t*>(base + L.rows);
  a.max_tiles = moe_route_max_tiles(r->T, r->E, r->k, r->block_m);
  a.timeout_ns = timeout_ns();
  return a;
}

// ids_given: the chosen experts and weights are already in r->ids / r->w (the
// fused router wrote them); logits are then not read.
moe_status route_impl(const float* logits, const moe_route_out* r, void* ws, size_t ws_bytes,
                      cudaStream_t s, int ids_given = 0) {
  moe_status st = check_route_out(r);
  if (st != MOE_OK) return st;
  if ((!ids_given && !logits && r->T > 0) || !ws) return MOE_ERR_ARG;
  if (!aligned16(logits) || !aligned16(ws)) return MOE_ERR_ALIGN;
  if (ws_bytes < route_ws_layout(r->T, r->E, r->k).total) return MOE_ERR_WORKSPACE;
  DevInfo di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  RouteArgs a = make_route_args(logits, r, ws);
  a.ids_given = ids_given;
  stage_mark(0, s);
  if (launch_route(a, s) != cudaSuccess) return MOE_ERR_CUDA;
  stage_mark(1, s);
  stage_mark(2, s);   // (routing is one step: stages 1 and 2 coincide)
  return MOE_OK;
}

// Batches of at most this many tokens take the decode path (split-K CUDA-core
// kernels); process-wide, changed by moe_debug_set_decode_max_t.
std::atomic<int> g_decode_max_t{kDecodeAutoT};

// path: 0 = by batch size, 1 = decode kernels, 2 = tensor-core grouped GEMM
moe_status ffn_impl(const uint16_t* x, int32_t T, int32_t d, const moe_q4_packed* W,
                    const moe_route_out* r, uint16_t* y, void* ws, size_t ws_bytes,
                    cudaStream_t s, int path = 0) {
  moe_status st = check_route_out(r);
  if (st != MOE_OK) return st;
  if ((st = check_packed(W)) != MOE_OK) return st;
  if ((T > 0 && (!x || !y)) || !ws) return MOE_ERR_ARG;   // x, y may be NULL when T == 0
  if (!aligned16(x) || !aligned16(y) || !aligned16(ws)) return MOE_ERR_ALIGN;
  if (T != r->T || d != W->d || W->E != r->E) return MOE_ERR_SHAPE;
  const PackLayout P = pack_layout(W->E, W->d, W->f, W->f_s);
  const uint8_t* pk = static_cast<const uint8_t*>(W->data);
  const int k = r->k, E = W->E, f = W->f, fs = W->f_s;
  const int max_tiles = moe_route_max_tiles(T, E, k, r->block_m);
  const FfnWs L = ffn_ws_layout(T, k, d, f, fs, max_tiles);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  DevInfo di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;

  char* base = static_cast<char*>(ws);
  const bool decode_fits = T <= kDecodeMaxT && decode_gu_bytes(T, k, d, f, fs) <= L.act_sh - L.act;
  if (path == 1 && !decode_fits) return MOE_ERR_SHAPE;
  if (path == 1 || (path == 0 && decode_fits && T <= g_decode_max_t.load())) {
    DecodeArgs a{};
    a.T = T;
    a.k = k;
    a.E = E;
    a.d = d;
    a.f = f;
    a.f_s = fs;
    a.f_max = f > fs ? f : fs;
    a.x = x;
    a.tiles = r->tiles;
    a.n_tiles = r->n_tiles;
    a.max_tiles = max_tiles;
    a.n_sh_tiles = fs ? (T + kDecTileRows - 1) / kDecTileRows : 0;
    a.perm = r->perm;
    a.wts = r->w;
    a.n_fb = P.gu.units;
    a.n_fb_sh = P.sgu.units;
    a.n_fb_max = a.n_fb > a.n_fb_sh ? a.n_fb : a.n_fb_sh;
    a.pk_gu = pk + P.gu.offset;
    a.pk_gu_sh = pk + P.sgu.offset;
    a.pk_dn = pk + P.dn.offset;
    a.pk_dn_sh = pk + P.sdn.offset;
    a.gu_part = reinterpret_cast<float*>(base + L.act);
    a.n_slots = T * k + T;
    a.y_acc = reinterpret_cast<float*>(base + L.y_acc);
    a.y = y;
    a.err = r->err;
    if (launch_decode(a, di.sms, s) != cudaSuccess) return MOE_ERR_CUDA;
    stage_mark(4, s);
    stage_mark(5, s);
    return MOE_OK;
  }
  uint16_t* act = reinterpret_cast<uint16_t*>(base + L.act);
  uint16_t* act_sh = reinterpret_cast<uint16_t*>(base + L.act_sh);
  const uint64_t act_rows = act_rows_capacity(T, k, max_tiles);
  const int tile_rows = gemm_tile_rows(r->block_m);
  // the shared activation rows are allocated up to a multiple of 128 (either tile height)
  const uint64_t act_sh_rows = (static_cast<uint64_t>(T) + 127) / 128 * 128;
  GemmArgs a{};
  a.E = E;
  a.T = T;
  a.k = k;
  a.d = d;
  a.f = f;
  a.f_s = fs;
  a.tiles = r->tiles;
  a.n_tiles = r->n_tiles;
  a.max_tiles = max_tiles;
  a.perm = r->perm;
  a.wts = r->w;
  a.y_acc = reinterpret_cast<float*>(base + L.y_acc);
  a.y = y;
  a.gbar = reinterpret_cast<int32_t*>(base + L.ctr);
  a.err = r->err;
  a.timeout_ns = timeout_ns();
  a.prefetch_guess = static_cast<long long>(T) * k <= 32ll * E;
  const int n_sh_tiles = fs ? (T + tile_rows - 1) / tile_rows : 0;

  const CUtensorMapSwizzle SW128 = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapDataType BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;

  // ---- pass 0: gate/up + SwiGLU
  {
    GemmArgs g = a;
    GemmMaps m;
    g.K = d;
    g.K_sh = d;
    g.n_fb = P.gu.units;
    g.n_fb_sh = P.sgu.units;
    g.n_sh_tiles = n_sh_tiles;
    g.pk = pk + P.gu.offset;
    g.pk_sh = pk + P.sgu.offset;
    bool ok = encode_2d(&m.B, BF16, 2, x, d, T, 64, 1, SW128) &&
              encode_2d(&m.C, BF16, 2, act, f, act_rows, 64, 16, SW128);
    if (fs) ok = ok && encode_2d(&m.C_sh, BF16, 2, act_sh, fs, act_sh_rows, 64, 16, SW128);
    else m.C_sh = m.C;
    m.B_sh = m.B;
    if (!ok) return MOE_ERR_CUDA;
    if (launch_gemm(0, tile_rows, g, m, di.sms, s) != cudaSuccess) return MOE_ERR_CUDA;
    stage_mark(3, s);
  }
  // ---- pass 1: down + weighted combine (+ shared expert)
  {
    GemmArgs g = a;
    GemmMaps m;
    g.K = f;
    g.K_sh = fs;
    g.n_fb = P.dn.units;
    g.n_fb_sh = P.sdn.units;
    g.n_sh_tiles = n_sh_tiles;
    g.pk = pk + P.dn.offset;
    g.pk_sh = pk + P.sdn.offset;
    bool ok = encode_2d(&m.B, BF16, 2, act, f, act_rows, 64, 16, SW128);
    if (fs) ok = ok && encode_2d(&m.B_sh, BF16, 2, act_sh, fs, act_sh_rows, 64, 16, SW128);
    else m.B_sh = m.B;
    m.C = m.B;
    m.C_sh = m.B_sh;
    if (!ok) return MOE_ERR_CUDA;
    if (launch_gemm(1, tile_rows, g, m, di.sms, s) != cudaSuccess) return MOE_ERR_CUDA;
    stage_mark(4, s);
  }
  stage_mark(5, s);   // (y is written by the down pass: stages 4 and 5 coincide)
  return MOE_OK;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// defer_weights: leave the chosen logits in r->w for the routing kernel (mode 2)
moe_status router_impl(const uint16_t* x, const uint16_t* w_router, int32_t T, int32_t d,
                       float* logits, const moe_route_out* r, cudaStream_t s,
                       bool defer_weights = false) {
  moe_status st = check_route_out(r);
  if (st != MOE_OK) return st;
  if (T != r->T) return MOE_ERR_SHAPE;
  if (r->E % 16 || r->E > kRouterMaxE || r->k > kRouterMaxK) return MOE_ERR_SHAPE;
  if (d < 64 || d % 64 || d > 16384) return MOE_ERR_SHAPE;
  if (T > 0 && (!x || !w_router)) return MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(logits)) return MOE_ERR_ALIGN;
  DevInfo di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  if (T == 0) return MOE_OK;
  RouterArgs a{};
  a.T = T;
  a.d = d;
  a.E = r->E;
  a.k = r->k;
  router_geometry(a);
  CUtensorMap mx, mw;
  const CUtensorMapSwizzle SW128 = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapDataType BF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!encode_2d(&mx, BF16, 2, x, d, T, 64, 128, SW128) ||
      !encode_2d(&mw, BF16, 2, w_router, d, r->E, 64, a.En, SW128))
    return MOE_ERR_CUDA;
  a.logits = logits;
  a.ids = r->ids;
  a.w = r->w;
  a.err = r->err;
  a.timeout_ns = timeout_ns();
  a.defer_weights = defer_weights ? 1 : 0;
  stage_mark(6, s);
  if (launch_router(a, mx, mw, s) != cudaSuccess) return MOE_ERR_CUDA;
  stage_mark(7, s);
  return MOE_OK;
}

// ---- fixed scratch for moe_route_noalloc (no counterpart on the pages)
constexpr int kNoAllocMaxT = 8192;
constexpr int kNoAllocMaxE = 256;
constexpr int kNoAllocMaxK = 8;
// routing scratch at the limits: the 4-byte count rows of 1024 blocks (8192
// tokens in blocks of at least 8) x 256 experts
constexpr size_t kNoAllocBytes = 4 * 1024 * 256;
__device__ __align__(256) unsigned char g_route_scratch[kNoAllocBytes];

// Device address of g_route_scratch on the current device, looked up once per
// device with that device current (host code cannot use the symbol itself).
moe_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> g(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return MOE_OK;
}

std::mutex g_ev_mu;
cudaEvent_t g_events[8] = {};
std::atomic<int> g_nevents{0};

}  // namespace

void stage_mark(int i, cudaStream_t s) {
  if (g_nevents.load(std::memory_order_relaxed) == 0) return;   // the common case: no timing requested
  std::lock_guard<std::mutex> g(g_ev_mu);
  if (i < g_nevents.load(std::memory_order_relaxed) && g_events[i]) cudaEventRecord(g_events[i], s);
}

}  // namespace moeq4

using namespace moeq4;

extern "C" {

int32_t moe_route_max_tiles(int32_t T, int32_t E, int32_t k, int32_t block_m) {
  if (T < 0 || E < 1 || k < 1 || block_m < 1) return 0;
  const long long rows = static_cast<long long>(T) * k;
  const long long n = rows / block_m + (rows < E ? rows : E);
  return static_cast<int32_t>(n);
}

size_t moe_route_workspace_size(int32_t T, int32_t E, int32_t k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  return route_ws_layout(T, E, k).total;
}

size_t moe_ffn_workspace_size(int32_t T, int32_t E, int32_t k, int32_t d, int32_t f,
                              int32_t f_s, int32_t block_m) {
  if (T < 0 || E < 1 || k < 1 || d < 1 || f < 1 || f_s < 0 || block_m < 1) return 0;
  return ffn_ws_layout(T, k, d, f, f_s, moe_route_max_tiles(T, E, k, block_m)).total;
}

size_t moe_layer_workspace_size(int32_t T, int32_t E, int32_t k, int32_t d, int32_t f,
                                int32_t f_s, int32_t block_m) {
  const size_t a = moe_route_workspace_size(T, E, k);
  const size_t b = moe_ffn_workspace_size(T, E, k, d, f, f_s, block_m);
  if (!a || !b) return 0;
  return align256(a) + b;
}

size_t moe_q4_packed_size(int32_t E, int32_t d, int32_t f, int32_t f_s) {
  if (check_dims(E, d, f, f_s) != MOE_OK) return 0;
  return pack_layout(E, d, f, f_s).total;
}

moe_status moe_q4_prepack(const moe_q4_weights* W, void* dst, size_t dst_bytes, void* stream) {
  moe_status st = check_weights(W);
  if (st != MOE_OK) return st;
  if (!dst) return MOE_ERR_ARG;
  if (!aligned16(dst)) return MOE_ERR_ALIGN;
  const PackLayout P = pack_layout(W->E, W->d, W->f, W->f_s);
  if (dst_bytes < P.total) return MOE_ERR_WORKSPACE;
  DevInfo di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* o = static_cast<uint8_t*>(dst);
  const int E = W->E, d = W->d, f = W->f, fs = W->f_s;
  if (launch_prepack(W->gate_up.qw, W->gate_up.scale, W->gate_up.bias, E, 2 * f, d, 0, f,
                     o + P.gu.offset, s) != cudaSuccess ||
      launch_prepack(W->down.qw, W->down.scale, W->down.bias, E, d, f, 1, d, o + P.dn.offset,
                     s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (fs > 0 &&
      (launch_prepack(W->sh_gate_up.qw, W->sh_gate_up.scale, W->sh_gate_up.bias, 1, 2 * fs, d, 0,
                      fs, o + P.sgu.offset, s) != cudaSuccess ||
       launch_prepack(W->sh_down.qw, W->sh_down.scale, W->sh_down.bias, 1, d, fs, 1, d,
                      o + P.sdn.offset, s) != cudaSuccess))
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_route(const float* logits, const moe_route_out* out, void* ws, size_t ws_bytes,
                     void* stream) {
  return route_impl(logits, out, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

moe_status moe_expert_ffn(const uint16_t* x, int32_t T, int32_t d, const moe_q4_packed* W,
                          const moe_route_out* r, uint16_t* y, void* ws, size_t ws_bytes,
                          void* stream) {
  return ffn_impl(x, T, d, W, r, y, ws, ws_bytes, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer(const uint16_t* x, const float* logits, int32_t T, const moe_q4_packed* W,
                     const moe_route_out* r, uint16_t* y, void* ws, size_t ws_bytes,
                     void* stream) {
  if (!W || !r) return MOE_ERR_ARG;
  if (r->T != T) return MOE_ERR_SHAPE;
  const size_t need = moe_layer_workspace_size(T, r->E, r->k, W->d, W->f, W->f_s, r->block_m);
  if (!ws || need == 0 || ws_bytes < need) return MOE_ERR_WORKSPACE;
  const size_t rsz = align256(moe_route_workspace_size(T, r->E, r->k));
  moe_status st;
  // validate the FFN arguments before anything is enqueued
  if ((st = check_packed(W)) != MOE_OK) return st;
  if (T > 0 && (!x || !y)) return MOE_ERR_ARG;   // x, y (and logits) may be NULL when T == 0
  if (!aligned16(x) || !aligned16(y)) return MOE_ERR_ALIGN;
  if (W->E != r->E) return MOE_ERR_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = route_impl(logits, r, ws, rsz, s)) != MOE_OK) return st;
  return ffn_impl(x, T, W->d, W, r, y, static_cast<char*>(ws) + rsz, ws_bytes - rsz, s);
}

moe_status moe_expert_ffn_decode(const uint16_t* x, int32_t T, int32_t d,
                                 const moe_q4_packed* W, const moe_route_out* r, uint16_t* y,
                                 void* ws, size_t ws_bytes, void* stream) {
  return ffn_impl(x, T, d, W, r, y, ws, ws_bytes, static_cast<cudaStream_t>(stream), 1);
}

moe_status moe_debug_set_decode_max_t(int32_t t) {
  if (t < 0) return MOE_ERR_ARG;
  g_decode_max_t.store(t);
  return MOE_OK;
}

moe_status moe_router_topk(const uint16_t* x, const uint16_t* w_router, int32_t T, int32_t d,
                           float* logits, const moe_route_out* out, void* stream) {
  return router_impl(x, w_router, T, d, logits, out, static_cast<cudaStream_t>(stream));
}

moe_status moe_route_ids(const moe_route_out* out, void* ws, size_t ws_bytes, void* stream) {
  return route_impl(nullptr, out, ws, ws_bytes, static_cast<cudaStream_t>(stream), 1);
}

moe_status moe_layer_router(const uint16_t* x, const uint16_t* w_router, int32_t T,
                            const moe_q4_packed* W, float* logits, const moe_route_out* r,
                            uint16_t* y, void* ws, size_t ws_bytes, void* stream) {
  if (!W || !r) return MOE_ERR_ARG;
  if (r->T != T) return MOE_ERR_SHAPE;
  const size_t need = moe_layer_workspace_size(T, r->E, r->k, W->d, W->f, W->f_s, r->block_m);
  if (!ws || need == 0 || ws_bytes < need) return MOE_ERR_WORKSPACE;
  const size_t rsz = align256(moe_route_workspace_size(T, r->E, r->k));
  moe_status st;
  // validate everything before anything is enqueued
  if ((st = check_packed(W)) != MOE_OK) return st;
  if ((st = check_route_out(r)) != MOE_OK) return st;
  if (T > 0 && (!x || !y)) return MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(ws)) return MOE_ERR_ALIGN;
  if (W->E != r->E) return MOE_ERR_SHAPE;
  if (r->E % 16 || r->E > kRouterMaxE || r->k > kRouterMaxK) return MOE_ERR_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = router_impl(x, w_router, T, W->d, logits, r, s, true)) != MOE_OK) return st;
  if ((st = route_impl(nullptr, r, ws, rsz, s, 2)) != MOE_OK) return st;
  return ffn_impl(x, T, W->d, W, r, y, static_cast<char*>(ws) + rsz, ws_bytes - rsz, s);
}

moe_status moe_get_device_error(const int32_t* err, int32_t* code, void* stream) {
  if (!err || !code) return MOE_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  *code = v;
  return v ? MOE_ERR_DEVICE : MOE_OK;
}

moe_status moe_debug_noalloc_scratch(void** addr, size_t* bytes) {
  if (!addr || !bytes) return MOE_ERR_ARG;
  moe_status st = noalloc_scratch(addr);
  if (st != MOE_OK) return st;
  *bytes = kNoAllocBytes;
  return MOE_OK;
}

moe_status moe_debug_set_stage_events(void* const* events, int32_t n) {
  if (n < 0 || n > 8 || (n > 0 && !events)) return MOE_ERR_ARG;
  std::lock_guard<std::mutex> g(g_ev_mu);
  for (int i = 0; i < 8; ++i) g_events[i] = (i < n) ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  g_nevents.store(n);
  return MOE_OK;
}

moe_status moe_route_noalloc(const float* logits, const moe_route_out* out, void* stream) {
  moe_status st = check_route_out(out);
  if (st != MOE_OK) return st;
  if (out->T > kNoAllocMaxT || out->E > kNoAllocMaxE || out->k > kNoAllocMaxK)
    return MOE_ERR_TOO_LARGE;
  const RouteWs L = route_ws_layout(out->T, out->E, out->k);
  if (L.total > kNoAllocBytes) return MOE_ERR_TOO_LARGE;
  void* ws = nullptr;
  if ((st = noalloc_scratch(&ws)) != MOE_OK) return st;
  // the count rows may hold anything: each call writes every row it reads
  return route_impl(logits, out, ws, kNoAllocBytes, static_cast<cudaStream_t>(stream));
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported or inconsistent shape";
    case MOE_ERR_WORKSPACE: return "workspace missing or too small";
    case MOE_ERR_CUDA: return "CUDA call or kernel launch failed";
    case MOE_ERR_DEVICE: return "device error word is set";
    case MOE_ERR_UNSUPPORTED: return "device is not sm_103";
    case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
    case MOE_ERR_TOO_LARGE:
      return "sizes exceed the fixed scratch of moe_route_noalloc (T <= 8192, E <= 256, k <= 8)";
    default: return "unknown status";
  }
}

}  // extern "C"
