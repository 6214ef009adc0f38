// moe_api.cu -- the extern "C" boundary of libmoe.so (declared in include/moe.h).
//
// Host-side argument checks, the workspace plan, the per-device error word,
// the launch counter, optional per-stage CUDA-event timing, and the sequence of
// stage launches S1..S8 on the caller's stream.  No device memory is
// allocated here: all scratch comes from the caller's workspace.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/moe.h"
#include "device.cuh"
#include "internal.h"

namespace moe {

__device__ int g_error_word;  // per-device fault word, see moe_get_last_error

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int64_t> g_launches{0};

// Filled once per device under g_dev_mu; `ready` is published with a release
// store after sms and err are written, and read with an acquire load, so a
// thread that sees it set also sees both fields.
struct DeviceInfo {
  std::atomic<bool> ready{false};
  int sms = 0;
  int* err = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

DeviceInfo* device_info() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
  DeviceInfo& di = g_dev[d];
  if (!di.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!di.ready.load(std::memory_order_relaxed)) {
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess)
        return nullptr;
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
      di.sms = sms;
      di.err = static_cast<int*>(p);
      di.ready.store(true, std::memory_order_release);
    }
  }
  return &di;
}

// ------------------------------------------------------------------ profiling
struct ProfRec {
  int stage;
  cudaEvent_t a, b;
};
std::atomic<uint32_t> g_prof_mask{0};  // bit s: time stage s
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

struct StageTimer {
  int stage;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  StageTimer(int st, cudaStream_t str) : stage(st), s(str) {
    if (g_prof_mask.load(std::memory_order_relaxed) & (1u << st)) {
      std::lock_guard<std::mutex> lk(g_prof_mu);
      a = take_event();
      if (a) cudaEventRecord(a, s);
    }
  }
  ~StageTimer() {
    if (!a) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    cudaEvent_t b = take_event();
    if (!b) return;
    cudaEventRecord(b, s);
    g_prof.push_back({stage, a, b});
  }
};

// ------------------------------------------------------------------ plan
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Plan {
  int T, H, I, E, k, K, R, RT, nch, BN, max_items, Is, L;
  bool shared;      // fp8 shared expert fused into the grouped GEMMs (rows R..R+T)
  bool shared_bf16; // bf16 shared expert as dense GEMMs (LatentMoE)
  bool mx;          // MXFP4 routed experts
  bool blockwise;   // fp8 experts with 128 x 128 block scales
  int packed;       // expert weights in tile-major order (moe_pack_weights)
  int act;          // FFN1 activation: 0 SwiGLU, 1 SiTU
  bool fused;       // S7 in the FFN2 epilogue (MOE_F_FUSED_COMBINE, where honoured)
  bool gather;      // S4 quantises per token; the FFN1 producer gathers the rows
  bool tc_router;   // S1 on the tensor cores, S2 made exact (route.cu)
  int rsplit;       // K ranges of the tensor-core router GEMM (logits blocks)
  size_t acc;       // fused combine: fp32 [T, H] sum
  size_t logits, idx, tw, cc, cbase, ticket, cnt, off, perm, src, row_w, xscale, items, n_items, xq, h,
      hq, hs, y, z, zflag, yn, hsh, rwp, rxn, rwn, total;
};

int choose_bn(const moe_problem* p) {
  // tuning().tile_n overrides the choice with a tile height the weight format
  // has kernels for; any other value is ignored
  const int v = tuning().tile_n;
  const double avg = (double)p->T * p->top_k / (p->E > 0 ? p->E : 1);
  if (p->wfmt == MOE_W_FP8_E4M3_BLOCK128) {  // block-wise tiles keep sums in registers
    if (v == 32 || v == 64) return v;
    return avg <= 24.0 ? 32 : 64;
  }
  if (p->wfmt == MOE_W_MXFP4_E2M1_E8M0_B32) {  // block-scaled kernel tiles: 32, 64, 96 rows
    if (v == 32 || v == 64 || v == 96) return v;
    return avg <= 24.0 ? 32 : avg <= 48.0 ? 64 : 96;
  }
  if (v == 32 || v == 64 || v == 128 || v == 256) return v;
  // fp8 per-channel: 128-row tiles up to ~96 rows per expert, even when
  // experts hold far fewer rows (the MMAs read only the item's rows rounded
  // up to 16).  A tile's stage then carries 48 KB, so four stages fill the
  // shared memory, and four stages stream the weights fastest: T=512, H=8192,
  // I=2048, E=256 top-8, FFN1 1.22 ms with 128-row tiles vs 1.34 ms with
  // 32-row tiles and six stages, 1.23 ms with 64-row tiles and four stages,
  // 1.26 ms with five
  if (avg <= 96.0) return 128;
  return 256;
}

bool use_pair_gemm(const Plan& q);

// S1 on the tensor cores with S2 made exact unless tuning().router_tile picks
// a CUDA-core tile (1..4).  With small batches split into K ranges, the
// tensor-core path is the faster at every size measured (S1 + S2 on GB300,
// E=256, H=8192: T=1 22 vs 41 us, T=512 35 vs 61, T=2048 55 vs 237; E=896,
// H=7168, k=16: T=1 31 vs 44, T=512 58 vs 220).
bool use_tc_router(const moe_problem* p) {
  const int rt = tuning().router_tile;
  (void)p;
  return rt == 0 || rt == 6;
}

Plan make_plan(const moe_problem* p) {
  Plan q{};
  q.T = p->T;
  q.H = p->H;
  q.I = p->I;
  q.E = p->E;
  q.k = p->top_k;
  q.K = p->latent > 0 ? p->latent : p->H;
  q.R = p->T * p->top_k;
  q.Is = p->I_shared;
  q.L = p->latent;
  q.shared_bf16 = p->I_shared > 0 && (p->flags & MOE_F_SHARED_BF16);
  q.shared = p->I_shared > 0 && !q.shared_bf16;
  q.mx = p->wfmt == MOE_W_MXFP4_E2M1_E8M0_B32;
  q.blockwise = p->wfmt == MOE_W_FP8_E4M3_BLOCK128;
  q.packed = (p->flags & MOE_F_PACKED_WEIGHTS) ? 1 : 0;
  q.act = (p->flags & MOE_F_SITU) ? 1 : 0;
  q.RT = q.R + (q.shared ? p->T : 0);
  q.nch = num_chunks(p->T);
  q.BN = choose_bn(p);
  q.max_items = (q.R + q.BN - 1) / q.BN + q.E +
                (p->I_shared > 0 ? (p->T + q.BN - 1) / q.BN + 1 : 0) + 1;
  // the fused combine runs in the single-SM fp8 per-channel FFN2 epilogue
  q.fused = (p->flags & MOE_F_FUSED_COMBINE) && !q.L && !q.mx && !q.blockwise &&
            !q.shared_bf16 && !use_pair_gemm(q);
  // tuning().ffn1_gather: the fp8 per-channel FFN1 gathers its rows by token
  // and S4 writes one row per token.  Off by default.  Single SM: the
  // producer's 16-byte cp.async copies (8 per row and stage) and the proxy
  // fence before each stage's MMAs cost more than the smaller S4 saves (T=512,
  // H=8192, I=2048, E=256 top-8, 128-row tiles: FFN1 1.35 vs 1.22 ms, S4 10.0
  // vs 12.9 us; T=2048: 1.84 vs 1.28 ms).  SM pairs: four-row TMA gathers
  // (tile::gather4, 32 per stage and CTA); T=16384: FFN1 12.06 vs 3.70 ms, S4
  // 0.099 vs 0.225 ms; T=8192 skewed: FFN1 5.63 vs 1.55 ms.
  q.gather = !q.mx && !q.blockwise && tuning().ffn1_gather;
  q.tc_router = use_tc_router(p);
  q.rsplit = q.H % 64 == 0 ? dense_split_k(q.T, q.E, 3 * q.H) : 1;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t T = q.T, E = q.E, k = q.k, R = q.R, RT = q.RT;
  q.logits = take(T * E * 4 * (size_t)q.rsplit);  // the router GEMM's K ranges, when split
  q.idx = take(T * k * 4);
  q.tw = take(T * k * 4);
  q.cc = take(E * q.nch * 4);
  q.cbase = take(E * q.nch * 4);
  q.ticket = take(4);
  q.cnt = take(E * 4);
  q.off = take((E + 1) * 4);
  q.perm = take(T * k * 4);
  q.src = take(R * 4);
  q.row_w = take(RT * 4);
  q.xscale = take(RT * 4);
  q.items = take((size_t)q.max_items * 16);
  q.n_items = take(16);
  q.xq = take(RT * (size_t)q.K);
  q.h = take(RT * (size_t)q.I * 2);
  q.hq = take(RT * (size_t)q.I);
  q.hs = take(RT * 4);
  q.y = take(q.fused ? 0 : RT * (size_t)q.K * 2);
  q.acc = take(q.fused ? T * (size_t)q.K * 4 : 0);
  q.z = take(q.L ? T * (size_t)q.L * 2 : 0);
  q.zflag = take(q.L ? latent_down_flag_bytes(q.T, q.L) : 0);
  // tensor-core router: weight pieces [E][3H] bf16 and the norms (always
  // planned, so that moe_router_topk can take either path)
  q.rwp = take(E * 3 * (size_t)q.H * 2);
  q.rxn = take(T * 4);
  q.rwn = take(E * 4);
  q.yn = take(q.L ? T * (size_t)q.L * 2 : 0);
  q.hsh = take(q.shared_bf16 ? T * (size_t)q.Is * 2 : 0);
  q.total = o;
  return q;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// ------------------------------------------------------------------ checks
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

int check_problem(const moe_problem* p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  if (p->T < 0 || p->H <= 0 || p->I <= 0 || p->E <= 0 || p->top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (p->top_k > p->E || p->top_k > kMaxTopK || p->E > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (p->H % 128 || p->I % 128 || p->I_shared < 0 || p->I_shared % 128 || p->latent < 0 ||
      p->latent % 128)
    return MOE_ERR_INVALID_ARG;
  if (p->wfmt != MOE_W_FP8_E4M3_PER_CHANNEL && p->wfmt != MOE_W_MXFP4_E2M1_E8M0_B32 &&
      p->wfmt != MOE_W_FP8_E4M3_BLOCK128)
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)p->T * p->top_k > (1 << 30) || (int64_t)p->T * p->H > (int64_t)1 << 40)
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

namespace {

// Shapes this library runs on the GPU: fp8 experts with an optional fp8 shared
// expert (I_shared == I, fused into the grouped GEMMs), or the LatentMoE block
// (latent > 0, optional bf16 shared expert) with fp8 or MXFP4 experts, or
// MXFP4 experts on their own; block-wise fp8 wherever fp8 runs, with K and I at
// most 16384 (the block-wise epilogue keeps 128 scales per block row).
int check_supported(const moe_problem* p) {
  const bool mx = p->wfmt == MOE_W_MXFP4_E2M1_E8M0_B32;
  if (p->wfmt == MOE_W_FP8_E4M3_BLOCK128 &&
      ((p->latent > 0 ? p->latent : p->H) > 16384 || p->I > 16384))
    return MOE_ERR_UNSUPPORTED;
  const bool sb = p->I_shared > 0 && (p->flags & MOE_F_SHARED_BF16);
  const bool s8 = p->I_shared > 0 && !sb;
  if (p->latent > 0) {
    if (s8) return MOE_ERR_UNSUPPORTED;
    if (p->H % 256 || p->latent % 256) return MOE_ERR_UNSUPPORTED;
    // the exact down projection keeps a bf16 row of x and a column list in shared memory
    if (2 * (int64_t)p->H + 2 * (int64_t)p->latent > 160 * 1024) return MOE_ERR_UNSUPPORTED;
  } else {
    if (sb) return MOE_ERR_UNSUPPORTED;
    if (mx && s8) return MOE_ERR_UNSUPPORTED;
  }
  if (s8 && p->I_shared != p->I) return MOE_ERR_UNSUPPORTED;
  if (mx && (p->latent > 0 ? p->latent : p->H) % 256) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// The router bias: with softmax routing it is added to the logits; with
// sigmoid (noaux_tc) routing it is added to the scores for selection only.
bool sigmoid_routing(const moe_problem* p) { return (p->flags & MOE_F_SIGMOID_ROUTING) != 0; }
const float* logit_bias(const moe_problem* p, const float* b) {
  return ((p->flags & MOE_F_ROUTER_BIAS) && !sigmoid_routing(p)) ? b : nullptr;
}
const float* selection_bias(const moe_problem* p, const float* b) {
  return ((p->flags & MOE_F_ROUTER_BIAS) && sigmoid_routing(p)) ? b : nullptr;
}

#define MOE_TRY(expr)                 \
  do {                                \
    cudaError_t _e = (expr);          \
    if (_e != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

GroupedFfnArgs ffn_args(const Plan& q, void* ws, const void* xq, const float* xscale,
                        const float* row_w, const void* w13, const void* w13_scale,
                        const void* w2, const void* w2_scale, const void* sw13,
                        const void* sw13_scale, const void* sw2, const void* sw2_scale, void* y,
                        int rows_total, int* err) {
  GroupedFfnArgs a{};
  a.items = at<int4>(ws, q.items);
  a.n_items = at<int32_t>(ws, q.n_items);
  a.max_items = q.max_items;
  a.E = q.E;
  a.K = q.K;
  a.I = q.I;
  a.rows_total = rows_total;
  a.xq = xq;
  a.xscale = xscale;
  a.row_w = row_w;
  a.w13 = w13;
  a.w13_scale = static_cast<const float*>(w13_scale);
  a.w2 = w2;
  a.w2_scale = static_cast<const float*>(w2_scale);
  a.sw13 = sw13;
  a.sw13_scale = static_cast<const float*>(sw13_scale);
  a.sw2 = sw2;
  a.sw2_scale = static_cast<const float*>(sw2_scale);
  a.h = at<void>(ws, q.h);
  a.hq = at<void>(ws, q.hq);
  a.hs = at<float>(ws, q.hs);
  a.y = y;
  a.R = q.R;
  a.T = q.T;
  a.BN = q.BN;
  a.packed = q.packed;
  a.act = q.act;
  a.blockwise = q.blockwise ? 1 : 0;
  a.err = err;
  return a;
}

// Small batches build the permutation in one single-block launch
// (index_small_kernel); tuning().index_3pass forces the three-kernel path.
// One single-block index launch for small batches; from 512 tokens the count,
// multi-block scan and rank kernels are faster (T=512, E=256: index stage 17
// vs 20 us on GB300).
bool use_index_small(const Plan& q) {
  if (tuning().index_3pass) return false;
  return q.T < 512 && index_small_fits(q.T, q.E);
}

// Large batches (256-row tiles) run the grouped GEMMs on SM pairs;
// tuning().gemm_1cta forces the single-SM kernels.
bool use_pair_gemm(const Plan& q) {
  if (tuning().gemm_1cta) return false;
  return !q.blockwise && q.BN == 256 && q.K % 256 == 0;
}

int run_experts(const Plan& q, const GroupedFfnArgs& a, int rows_total, cudaStream_t s) {
  const bool pair = !q.mx && use_pair_gemm(q);
  {
    StageTimer t(MOE_STAGE_FFN1, s);
    MOE_TRY(q.mx ? launch_ffn1_mx(a, s) : pair ? launch_ffn1_pair(a, s) : launch_ffn1(a, s));
  }
  {
    StageTimer t(MOE_STAGE_REQUANT, s);
    MOE_TRY(launch_requant(a.h, a.hq, a.hs, rows_total, q.I, s));
  }
  {
    StageTimer t(MOE_STAGE_FFN2, s);
    MOE_TRY(q.mx ? launch_ffn2_mx(a, s) : pair ? launch_ffn2_pair(a, s) : launch_ffn2(a, s));
  }
  return MOE_OK;
}

// S1 + S2 into idx / tw [T, k]: tensor-core logits with the selection made
// exact, or the canonical CUDA-core router and top-k; the same routing either way.
int route_tokens(const moe_problem* p, const Plan& q, void* ws, const void* x,
                 const float* router_w, const float* router_bias, int32_t* idx, float* tw,
                 int* err, cudaStream_t s) {
  float* logits = at<float>(ws, q.logits);
  const int sig = sigmoid_routing(p) ? 1 : 0;
  if (q.tc_router) {
    {
      StageTimer t(MOE_STAGE_ROUTER, s);
      MOE_TRY(launch_router_tc(x, router_w, q.T, q.H, q.E, at<uint16_t>(ws, q.rwp),
                               at<float>(ws, q.rxn), at<float>(ws, q.rwn), logits, q.rsplit, err,
                               s));
    }
    StageTimer t(MOE_STAGE_TOPK, s);
    MOE_TRY(launch_topk_tc(logits, q.rsplit, logit_bias(p, router_bias),
                           selection_bias(p, router_bias), sig, x, router_w, at<float>(ws, q.rxn),
                           at<float>(ws, q.rwn), idx, tw, q.T, q.H, q.E, q.k, s));
    return MOE_OK;
  }
  {
    StageTimer t(MOE_STAGE_ROUTER, s);
    MOE_TRY(launch_router_logits(x, router_w, logit_bias(p, router_bias), logits, q.T, q.H, q.E,
                                 err, s));
  }
  StageTimer t(MOE_STAGE_TOPK, s);
  MOE_TRY(launch_topk(logits, selection_bias(p, router_bias), sig, idx, tw, q.T, q.E, q.k, s));
  return MOE_OK;
}

}  // namespace

int device_sm_count() {
  DeviceInfo* d = device_info();
  return d ? d->sms : 1;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

namespace {

// moe_tuning, field by field, so that readers never see a half-written set.
std::atomic<int32_t> g_tune[8];
std::once_flag g_tune_once;

bool env_is(const char* name, const char* value) {
  const char* v = std::getenv(name);
  return v && std::strcmp(v, value) == 0;
}

void tuning_from_env() {
  const char* tn = std::getenv("MOE_TILE_N");
  int rt = 0;
  if (env_is("MOE_ROUTER_TILE", "8x8")) rt = 1;
  if (env_is("MOE_ROUTER_TILE", "8x16")) rt = 2;
  if (env_is("MOE_ROUTER_TILE", "8x16s4")) rt = 3;
  if (env_is("MOE_ROUTER_TILE", "12w8x16")) rt = 4;
  if (env_is("MOE_ROUTER_TILE", "tc")) rt = 6;
  const int32_t v[8] = {tn ? std::atoi(tn) : 0,
                        env_is("MOE_GATHER", "1") ? 1 : 0,
                        env_is("MOE_INDEX", "3pass") ? 1 : 0,
                        env_is("MOE_GEMM", "1cta") ? 1 : 0,
                        env_is("MOE_PAIR_SMALL", "0") ? 0 : 1,
                        env_is("MOE_MX", "1cta") ? 1 : 0,
                        rt,
                        env_is("MOE_PDL", "0") ? 0 : 1};
  for (int i = 0; i < 8; ++i) g_tune[i].store(v[i], std::memory_order_relaxed);
}

}  // namespace

moe_tuning tuning() {
  std::call_once(g_tune_once, tuning_from_env);
  moe_tuning t;
  t.tile_n = g_tune[0].load(std::memory_order_relaxed);
  t.ffn1_gather = g_tune[1].load(std::memory_order_relaxed);
  t.index_3pass = g_tune[2].load(std::memory_order_relaxed);
  t.gemm_1cta = g_tune[3].load(std::memory_order_relaxed);
  t.pair_small = g_tune[4].load(std::memory_order_relaxed);
  t.mx_1cta = g_tune[5].load(std::memory_order_relaxed);
  t.router_tile = g_tune[6].load(std::memory_order_relaxed);
  t.pdl = g_tune[7].load(std::memory_order_relaxed);
  return t;
}

bool pdl_enabled() {
  std::call_once(g_tune_once, tuning_from_env);
  return g_tune[7].load(std::memory_order_relaxed) != 0;
}

int* device_error_word() {
  DeviceInfo* d = device_info();
  return d ? d->err : nullptr;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    default: return "MOE_ERR_UNKNOWN";
  }
}

int moe_describe(const moe_problem* p, char* buf, size_t len) {
  if (!buf || len == 0) return MOE_ERR_INVALID_ARG;
  buf[0] = 0;
  int st = check_problem(p);
  if (st) return st;
  st = check_supported(p);
  if (st) return st;
  const Plan q = make_plan(p);
  const bool pair = !q.mx && use_pair_gemm(q);
  GroupedFfnArgs mxa{};
  mxa.packed = q.packed;
  mxa.I = q.I;
  mxa.K = q.K;
  auto gemm = [&](bool ffn1) {
    if (q.mx) return mx_pair_eligible(mxa, ffn1) ? "grouped_mx_pair_kernel" : "grouped_mx_kernel";
    return pair ? "pair_gemm_kernel" : "grouped_ffn_kernel";
  };
  char router[48];
  if (q.tc_router)
    std::snprintf(router, sizeof router, "tensor-cores,k_ranges=%d", q.rsplit);
  else
    std::snprintf(router, sizeof router, "cuda-cores");
  const int n = std::snprintf(
      buf, len,
      "ffn1=%s<FFN1,BN=%d> ffn2=%s<FFN2,BN=%d> tile_rows=%d ffn1_rows=%s weights=%s%s%s "
      "combine=%s router=%s max_items=%d workspace=%zu",
      gemm(true), q.BN, gemm(false), q.BN, q.BN, q.gather ? "gathered" : "permuted",
      q.mx ? "mxfp4" : q.blockwise ? "fp8-block128" : "fp8", q.packed ? ",packed" : "",
      q.L > 0 ? " latent=bf16-pair-gemms" : "",
      q.fused ? "fused-ffn2-fp32-sum" : q.L > 0 ? "gather-rmsnorm" : "gather", router,
      q.max_items, q.total);
  return (n < 0 || (size_t)n >= len) ? MOE_ERR_INVALID_ARG : MOE_OK;
}

size_t moe_workspace_bytes(const moe_problem* p) {
  if (check_problem(p) != MOE_OK) return 0;
  return make_plan(p).total;
}

int moe_router_logits(const moe_problem* p, const void* x, const float* router_w,
                      const float* bias, float* logits, void* stream) {
  int st = check_problem(p);
  if (st) return st;
  if (!x || !router_w || !logits) return MOE_ERR_INVALID_ARG;
  if ((p->flags & MOE_F_ROUTER_BIAS) && !bias) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(router_w, 16)) return MOE_ERR_INVALID_ARG;
  if (p->T == 0) return MOE_OK;
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StageTimer t(MOE_STAGE_ROUTER, s);
  return cuda_status(launch_router_logits(x, router_w, logit_bias(p, bias), logits, p->T, p->H,
                                          p->E, di->err, s));
}

int moe_route(const moe_problem* p, const float* logits, const float* bias, int32_t* topk_idx,
              float* topk_w, void* stream) {
  int st = check_problem(p);
  if (st) return st;
  if (!logits || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if (sigmoid_routing(p) && (p->flags & MOE_F_ROUTER_BIAS) && !bias) return MOE_ERR_INVALID_ARG;
  if (p->T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StageTimer t(MOE_STAGE_TOPK, s);
  return cuda_status(launch_topk(logits, selection_bias(p, bias), sigmoid_routing(p) ? 1 : 0,
                                 topk_idx, topk_w, p->T, p->E, p->top_k, s));
}

int moe_router_topk(const moe_problem* p, const void* x, const float* router_w,
                    const float* bias, int32_t* topk_idx, float* topk_w, void* ws,
                    size_t ws_bytes, void* stream) {
  int st = check_problem(p);
  if (st) return st;
  if (!x || !router_w || !topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
  if ((p->flags & MOE_F_ROUTER_BIAS) && !bias) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(router_w, 16)) return MOE_ERR_INVALID_ARG;
  const Plan q = make_plan(p);
  if (!ws || ws_bytes < q.total || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  if (p->T == 0) return MOE_OK;
  return route_tokens(p, q, ws, x, router_w, bias, topk_idx, topk_w, di->err,
                      static_cast<cudaStream_t>(stream));
}

int moe_permute(const moe_problem* p, const int32_t* topk_idx, const void* x, int32_t* counts,
                int32_t* offsets, int32_t* perm, int32_t* src_row, void* xq_perm,
                float* xscale_perm, void* ws, size_t ws_bytes, void* stream) {
  int st = check_problem(p);
  if (st) return st;
  if (!topk_idx || !x || !counts || !offsets || !perm || !src_row || !xq_perm || !xscale_perm)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(xq_perm, 16)) return MOE_ERR_INVALID_ARG;
  const Plan q = make_plan(p);
  if (!ws || ws_bytes < q.total || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  if (p->T == 0) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MOE_TRY(cudaMemsetAsync(counts, 0, sizeof(int32_t) * p->E, s));
    MOE_TRY(cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (p->E + 1), s));
    return MOE_OK;
  }
  const int K = q.K;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    StageTimer t(MOE_STAGE_INDEX, s);
    if (use_index_small(q)) {
      MOE_TRY(launch_index_small(topk_idx, nullptr, counts, offsets, perm, src_row, nullptr, q.T,
                                 q.E, q.k, nullptr, nullptr, 0, q.BN, 0, 0, di->err, s));
    } else {
      MOE_TRY(launch_count(topk_idx, at<int32_t>(ws, q.cc), at<int32_t>(ws, q.ticket), q.T, q.E,
                           q.k, di->err, s));
      MOE_TRY(launch_scan(at<int32_t>(ws, q.cc), at<int32_t>(ws, q.cbase), counts, offsets,
                          at<int32_t>(ws, q.ticket), q.T, q.E, q.k, nullptr, nullptr, 0, q.BN, 0,
                          0, s));
      MOE_TRY(launch_rank(topk_idx, nullptr, offsets, at<int32_t>(ws, q.cbase), perm, src_row,
                          nullptr, q.T, q.E, q.k, s));
    }
  }
  {
    StageTimer t(MOE_STAGE_SCATTER, s);
    MOE_TRY(launch_quant_scatter(x, perm, xq_perm, xscale_perm, q.T, K, q.k, -1, di->err, s));
  }
  return MOE_OK;
}

int moe_expert_ffn(const moe_problem* p, const int32_t* offsets, const void* xq_perm,
                   const float* xscale_perm, const float* row_w, const void* w13,
                   const void* w13_scale, const void* w2, const void* w2_scale, void* y,
                   void* ws, size_t ws_bytes, void* stream) {
  int st = check_problem(p);
  if (st) return st;
  if (!offsets || !xq_perm || !xscale_perm || !w13 || !w13_scale || !w2 || !w2_scale || !y)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(xq_perm, 16) || !aligned(w13, 32) || !aligned(w2, 32) || !aligned(y, 16) ||
      !aligned(w13_scale, 4) || !aligned(w2_scale, 4))
    return MOE_ERR_INVALID_ARG;
  st = check_supported(p);
  if (st) return st;
  const Plan q = make_plan(p);
  if (!ws || ws_bytes < q.total || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  if (p->T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    StageTimer t(MOE_STAGE_INDEX, s);
    MOE_TRY(launch_items_from_offsets(offsets, q.E, at<int4>(ws, q.items),
                                      at<int32_t>(ws, q.n_items), q.max_items, q.BN, s));
  }
  GroupedFfnArgs a = ffn_args(q, ws, xq_perm, xscale_perm, row_w, w13, w13_scale, w2, w2_scale,
                              nullptr, nullptr, nullptr, nullptr, y, q.R, di->err);
  return run_experts(q, a, q.R, s);
}

int moe_latent_down(const moe_problem* p, const void* x, const void* latent_down, void* z,
                    void* ws, size_t ws_bytes, void* stream) {
  int st = check_problem(p);
  if (st) return st;
  if (p->latent <= 0 || !x || !latent_down || !z) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(latent_down, 16) || !aligned(z, 16)) return MOE_ERR_INVALID_ARG;
  st = check_supported(p);
  if (st) return st;
  const Plan q = make_plan(p);
  if (!ws || ws_bytes < q.total || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  if (p->T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StageTimer t(MOE_STAGE_LATENT_DOWN, s);
  return cuda_status(launch_latent_down(x, latent_down, z, at<uint32_t>(ws, q.zflag), q.T, q.H,
                                        q.L, di->err, s));
}

int moe_unpermute(const moe_problem* p, const void* y_rows, const int32_t* perm,
                  const void* shared, void* out, void* stream) {
  int st = check_problem(p);
  if (st) return st;
  if (!y_rows || !perm || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(y_rows, 16) || !aligned(out, 16) || (shared && !aligned(shared, 16)))
    return MOE_ERR_INVALID_ARG;
  if (p->T == 0) return MOE_OK;
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  StageTimer t(MOE_STAGE_COMBINE, s);
  return cuda_status(launch_combine(y_rows, perm, shared, out, p->T, p->H, p->top_k, di->err, s));
}

int moe_forward(const moe_problem* p, const void* x, const float* router_w,
                const float* router_bias, const void* w13, const void* w13_scale,
                const void* w2, const void* w2_scale, const void* shared_w13,
                const void* shared_w13_scale, const void* shared_w2,
                const void* shared_w2_scale, const void* latent_down, const void* latent_up,
                const void* latent_gamma, void* out, void* ws, size_t ws_bytes, void* stream) {
  int st = check_problem(p);
  if (st) return st;
  if (!x || !router_w || !w13 || !w13_scale || !w2 || !w2_scale || !out) return MOE_ERR_INVALID_ARG;
  if ((p->flags & MOE_F_ROUTER_BIAS) && !router_bias) return MOE_ERR_INVALID_ARG;
  if (p->I_shared > 0 && (!shared_w13 || !shared_w2)) return MOE_ERR_INVALID_ARG;
  if (p->I_shared > 0 && !(p->flags & MOE_F_SHARED_BF16) && (!shared_w13_scale || !shared_w2_scale))
    return MOE_ERR_INVALID_ARG;
  if (p->latent > 0 && (!latent_down || !latent_up || !latent_gamma)) return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(router_w, 16) || !aligned(w13, 32) || !aligned(w2, 32) ||
      !aligned(out, 16) || (shared_w13 && !aligned(shared_w13, 16)) ||
      (shared_w2 && !aligned(shared_w2, 16)) || (latent_down && !aligned(latent_down, 16)) ||
      (latent_up && !aligned(latent_up, 16)) || (latent_gamma && !aligned(latent_gamma, 16)) ||
      !aligned(w13_scale, 4) || !aligned(w2_scale, 4))
    return MOE_ERR_INVALID_ARG;
  st = check_supported(p);
  if (st) return st;
  const Plan q = make_plan(p);
  if (!ws || ws_bytes < q.total || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  if (p->T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t* idx = at<int32_t>(ws, q.idx);
  float* tw = at<float>(ws, q.tw);
  int32_t* off = at<int32_t>(ws, q.off);
  int32_t* perm = at<int32_t>(ws, q.perm);
  float* row_w = at<float>(ws, q.row_w);
  float* xscale = at<float>(ws, q.xscale);
  uint8_t* xq = at<uint8_t>(ws, q.xq);
  uint16_t* y = at<uint16_t>(ws, q.y);
  st = route_tokens(p, q, ws, x, router_w, router_bias, idx, tw, di->err, s);
  if (st) return st;
  // LatentMoE: the experts run on z = bf16(x Wd^T) ("Kimi K3 ...", s.2.4)
  const void* xin = x;
  if (q.L) {
    StageTimer t(MOE_STAGE_LATENT_DOWN, s);
    MOE_TRY(launch_latent_down(x, latent_down, at<void>(ws, q.z), at<uint32_t>(ws, q.zflag), q.T,
                               q.H, q.L, di->err, s));
    xin = at<void>(ws, q.z);
  }
  {
    StageTimer t(MOE_STAGE_INDEX, s);
    if (use_index_small(q)) {
      MOE_TRY(launch_index_small(idx, tw, at<int32_t>(ws, q.cnt), off, perm, at<int32_t>(ws, q.src),
                                 row_w, q.T, q.E, q.k, at<int4>(ws, q.items),
                                 at<int32_t>(ws, q.n_items), q.max_items, q.BN, q.R,
                                 q.shared ? q.T : 0, di->err, s));
    } else {
      MOE_TRY(launch_count(idx, at<int32_t>(ws, q.cc), at<int32_t>(ws, q.ticket), q.T, q.E, q.k,
                           di->err, s));
      MOE_TRY(launch_scan(at<int32_t>(ws, q.cc), at<int32_t>(ws, q.cbase), at<int32_t>(ws, q.cnt),
                          off, at<int32_t>(ws, q.ticket), q.T, q.E, q.k, at<int4>(ws, q.items),
                          at<int32_t>(ws, q.n_items), q.max_items, q.BN, q.R, q.shared ? q.T : 0,
                          s));
      MOE_TRY(launch_rank(idx, tw, off, at<int32_t>(ws, q.cbase), perm, at<int32_t>(ws, q.src),
                          row_w, q.T, q.E, q.k, s));
    }
  }
  {
    StageTimer t(MOE_STAGE_SCATTER, s);
    if (q.gather)  // one fp8 row per token (rows 0..T-1 of xq); FFN1 gathers them
      MOE_TRY(launch_quant_scatter(xin, nullptr, xq, xscale, q.T, q.K, 0, 0, di->err, s,
                                   q.fused ? at<float>(ws, q.acc) : nullptr));
    else
      MOE_TRY(launch_quant_scatter(xin, perm, xq, xscale, q.T, q.K, q.k, q.shared ? q.R : -1,
                                   di->err, s, q.fused ? at<float>(ws, q.acc) : nullptr));
  }
  GroupedFfnArgs a = ffn_args(q, ws, xq, xscale, row_w, w13, w13_scale, w2, w2_scale, shared_w13,
                              shared_w13_scale, shared_w2, shared_w2_scale, y, q.RT, di->err);
  a.src = at<int32_t>(ws, q.src);
  a.gather = q.gather ? 1 : 0;
  if (q.fused) a.out_acc = at<float>(ws, q.acc);
  st = run_experts(q, a, q.RT, s);
  if (st) return st;
  if (q.fused) {
    StageTimer t(MOE_STAGE_COMBINE, s);
    MOE_TRY(launch_acc_to_bf16(at<float>(ws, q.acc), out, (size_t)q.T * q.H, s));
    return MOE_OK;
  }
  if (!q.L) {
    StageTimer t(MOE_STAGE_COMBINE, s);
    MOE_TRY(launch_combine(y, perm, q.shared ? y + (size_t)q.R * q.H : nullptr, out, q.T, q.H, q.k,
                           di->err, s));
    return MOE_OK;
  }
  // LatentMoE tail: RMSNorm of the routed combine, bf16 shared expert on the
  // raw hidden, and out = bf16(yn Wu^T + h_s W2s^T) in one accumulation.
  {
    StageTimer t(MOE_STAGE_COMBINE, s);
    MOE_TRY(launch_combine_rmsnorm(y, perm, latent_gamma, at<void>(ws, q.yn), q.T, q.L, q.k, 1e-6f,
                                   di->err, s));
  }
  if (q.shared_bf16) {
    StageTimer t(MOE_STAGE_SHARED, s);
    DenseGemmArgs d{};
    d.x = x;
    d.w = shared_w13;
    d.K1 = q.H;
    d.rows = q.T;
    d.N = q.Is;
    d.swiglu = true;
    d.act = q.act;
    d.out = at<void>(ws, q.hsh);
    d.err = di->err;
    MOE_TRY(launch_dense_bf16(d, s));
  }
  {
    StageTimer t(MOE_STAGE_LATENT_UP, s);
    DenseGemmArgs d{};
    d.x = at<void>(ws, q.yn);
    d.w = latent_up;
    d.K1 = q.L;
    if (q.shared_bf16) {
      d.x2 = at<void>(ws, q.hsh);
      d.w2 = shared_w2;
      d.K2 = q.Is;
    }
    d.rows = q.T;
    d.N = q.H;
    d.out = out;
    d.err = di->err;
    MOE_TRY(launch_dense_bf16(d, s));
  }
  return MOE_OK;
}

int moe_get_last_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  DeviceInfo* di = device_info();
  if (!di) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, di->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (v != 0) {
    int zero = 0;
    if (cudaMemcpy(di->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  return v;
}

int64_t moe_launch_count(void) { return g_launches.load(); }

int moe_get_tuning(moe_tuning* t) {
  if (!t) return MOE_ERR_INVALID_ARG;
  *t = tuning();
  return MOE_OK;
}

int moe_set_tuning(const moe_tuning* t) {
  if (!t) return MOE_ERR_INVALID_ARG;
  const int32_t v[8] = {t->tile_n, t->ffn1_gather, t->index_3pass, t->gemm_1cta,
                        t->pair_small, t->mx_1cta, t->router_tile, t->pdl};
  const bool tile_ok = v[0] == 0 || v[0] == 32 || v[0] == 64 || v[0] == 96 || v[0] == 128 ||
                       v[0] == 256;
  if (!tile_ok || v[6] < 0 || v[6] > 6 || v[6] == 5) return MOE_ERR_INVALID_ARG;
  for (int i : {1, 2, 3, 4, 5, 7})
    if (v[i] != 0 && v[i] != 1) return MOE_ERR_INVALID_ARG;
  std::call_once(g_tune_once, tuning_from_env);  // the environment never overrides a set
  for (int i = 0; i < 8; ++i) g_tune[i].store(v[i], std::memory_order_relaxed);
  return MOE_OK;
}

int moe_profile_enable(int mask) {
  g_prof_mask.store(static_cast<uint32_t>(mask));
  return MOE_OK;
}

int moe_profile_read(double* stage_ms, int64_t* stage_launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (int i = 0; i < MOE_STAGE_COUNT; ++i) {
    if (stage_ms) stage_ms[i] = 0.0;
    if (stage_launches) stage_launches[i] = 0;
  }
  int rc = MOE_OK;
  for (const ProfRec& r : g_prof) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      rc = MOE_ERR_CUDA;
    if (r.stage >= 0 && r.stage < MOE_STAGE_COUNT) {
      if (stage_ms) stage_ms[r.stage] += ms;
      if (stage_launches) stage_launches[r.stage] += 1;
    }
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_prof.clear();
  return rc;
}

}  // extern "C"
