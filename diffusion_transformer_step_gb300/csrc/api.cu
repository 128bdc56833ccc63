// The C ABI (include/dit.h): argument validation, workspace layout, the launch
// sequence of a dual-stream block, a single-stream block and the whole step, and the
// host runtime pieces (launch accounting, per-launch timing, TMA descriptor encoding).
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/dit.h"
#include "runtime.h"

namespace dit {

// ---------------------------------------------------------------------------------
// Launch accounting and timing
// ---------------------------------------------------------------------------------
namespace {
std::atomic<unsigned long long> g_launches{0};
// While this thread captures a step into a graph, its launches do not run: they are
// counted here instead and added to g_launches each time the graph is replayed.  Per
// thread, so that launches other threads issue meanwhile are counted as usual.
thread_local bool t_capturing = false;
thread_local unsigned long long t_captured = 0;
std::mutex g_timing_mu;
bool g_timing_on = false;
unsigned int g_timing_mask = ~0u;  // classes whose launches get an event pair
struct TimingRec {
  int cls;
  cudaEvent_t start, stop;
};
std::vector<TimingRec> g_recs;
int g_rec_used = 0;
}  // namespace

const char* kernel_class_name(int cls) {
  static const char* names[kClsCount] = {
      "adaln",          "gemm_qkv_rmsnorm_rope", "gemm_fused_qkv_mlp",  "gemm_gated_residual",
      "gemm_swiglu",    "gemm_plain",            "attention",           "modulation_gemv",
      "rope_table",     "pack_mlp_in",           "gemm_dual_out_proj",  "gemm_dual_mlp_out",
      "gemm_single_out_proj", "quantize_act"};
  return (cls >= 0 && cls < kClsCount) ? names[cls] : "?";
}

LaunchScope::LaunchScope(int cls, cudaStream_t stream) : slot_(-1), stream_(stream), captured_(t_capturing) {
  if (t_capturing)
    ++t_captured;
  else
    g_launches.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lk(g_timing_mu);
  if (g_timing_on && ((g_timing_mask >> cls) & 1u) && g_rec_used < (int)g_recs.size()) {
    slot_ = g_rec_used++;
    g_recs[slot_].cls = cls;
    record(g_recs[slot_].start);
  }
}

LaunchScope::~LaunchScope() {
  if (slot_ >= 0) record(g_recs[slot_].stop);
}

// While a step is being captured, the event pair becomes a pair of event-record nodes of
// the graph (re-recorded on every replay), so a replayed step can be timed per launch too.
void LaunchScope::record(cudaEvent_t e) {
  if (captured_)
    cudaEventRecordWithFlags(e, stream_, cudaEventRecordExternal);
  else
    cudaEventRecord(e, stream_);
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("DIT_NO_PDL");
    return !(e && e[0] == '1');
  }();
  return on;
}

int sm_count() {
  static std::atomic<int> cached[16];  // per device, filled by whichever host thread asks first
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 16) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev >= 0 && dev < 16) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

static bool encode_tmap_typed(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                              const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box);

bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap_typed(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes, box);
}

bool encode_tmap_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap_typed(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rank, dims, strides_bytes, box);
}

static bool encode_tmap_typed(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                              const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box) {
  typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                               const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                               CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  if (!fn) return false;
  cuuint64_t d[5];
  cuuint64_t st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
  const CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, st, bx,
                        es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------------
// Validation and workspace layout
// ---------------------------------------------------------------------------------
namespace {

constexpr int kMaxBatch = 64;
constexpr int kMaxDenoiseSteps = 8;
constexpr long long kMaxTokens = 1 << 20;

inline bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dit_status check_config(const dit_config* c) {
  if (!c) return DIT_ERR_INVALID_ARG;
  // hidden first (at most 4096), so that heads * 128 below cannot overflow; the GEMM widths
  // stay within dit_linear's limits
  if (!adaln_supports(c->hidden)) return DIT_ERR_UNSUPPORTED;
  if (c->head_dim != 128 || c->heads <= 0 || c->heads > c->hidden || c->hidden != c->heads * 128)
    return DIT_ERR_UNSUPPORTED;
  if (c->mlp_hidden <= 0 || c->mlp_hidden % 128 != 0 || c->mlp_hidden > kMaxTokens / 2) return DIT_ERR_UNSUPPORTED;
  if (c->in_channels <= 0 || c->in_channels % 32 != 0 || c->in_channels > kMaxTokens) return DIT_ERR_UNSUPPORTED;
  if (c->txt_dim <= 0 || c->txt_dim % 8 != 0 || c->txt_dim > kMaxTokens) return DIT_ERR_UNSUPPORTED;
  if (c->n_dual < 0 || c->n_single < 0) return DIT_ERR_INVALID_ARG;
  int sum = 0;
  for (int i = 0; i < 4; ++i) {
    if (c->axes_dim[i] < 0 || c->axes_dim[i] % 2 != 0) return DIT_ERR_UNSUPPORTED;
    sum += c->axes_dim[i];
  }
  if (sum != c->head_dim) return DIT_ERR_UNSUPPORTED;
  if (!(c->rope_theta > 0.f) || !(c->eps > 0.f)) return DIT_ERR_INVALID_ARG;
  return DIT_OK;
}

dit_status check_shape(const dit_shape* s) {
  if (!s) return DIT_ERR_INVALID_ARG;
  if (s->batch < 1 || s->batch > kMaxBatch) return DIT_ERR_INVALID_ARG;
  if (s->n_txt < 1 || s->n_img < 1 || s->n_ref < 0) return DIT_ERR_INVALID_ARG;
  if ((long long)s->n_txt + s->n_img + s->n_ref > kMaxTokens) return DIT_ERR_UNSUPPORTED;
  return DIT_OK;
}

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  size_t status, h1, h2, mod, x, x1, y, q, k, v, cat, yq, ascale, cq, cscale;
  size_t in_img, in_ref, in_txt, in_sigma, out_vel;
  size_t den_sigma, den_coef, den_mod, den_h1, den_h2, den_state, den_xbf;
  size_t block_end, step_end, total;
};

Layout layout(const dit_config& c, const dit_shape& s) {
  const size_t B = s.batch, N = (size_t)s.n_txt + s.n_img + s.n_ref, H = c.hidden, F = c.mlp_hidden;
  Layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = up256(o + bytes);
    return at;
  };
  L.status = take(sizeof(DeviceStatus));
  L.h1 = take(B * H * 4);
  L.h2 = take(B * H * 4);
  L.y = take(B * N * H * 2);
  L.q = take(B * N * H * 2);
  L.k = take(B * N * H * 2);
  L.v = take(B * N * H * 2);
  L.cat = take(B * N * (H + F) * 2);
  L.x1 = take(B * N * H * 4);
  L.yq = take(B * N * H);
  L.ascale = take(B * N * 4);
  L.cq = take(B * N * (H + F));  // e4m3 input of an out-projection (attention output / activations)
  L.cscale = take(B * N * 4);
  L.block_end = o;
  L.mod = take(B * 17 * H * 2);
  L.x = take(B * N * H * 2);
  L.step_end = o;
  L.in_img = take(B * (size_t)s.n_img * c.in_channels * 2);
  L.in_ref = take(B * (size_t)s.n_ref * c.in_channels * 2);
  L.in_txt = take(B * (size_t)s.n_txt * c.txt_dim * 2);
  L.in_sigma = take(B * 4);
  L.out_vel = take(B * (size_t)s.n_img * c.in_channels * 2);
  L.den_sigma = take((size_t)kMaxDenoiseSteps * B * 4);
  L.den_coef = take((size_t)kMaxDenoiseSteps * B * 4);
  L.den_mod = take((size_t)kMaxDenoiseSteps * B * 17 * H * 2);
  L.den_h1 = take((size_t)kMaxDenoiseSteps * B * H * 4);
  L.den_h2 = take((size_t)kMaxDenoiseSteps * B * H * 4);
  L.den_state = take(B * (size_t)s.n_img * c.in_channels * 4);
  L.den_xbf = take(B * (size_t)s.n_img * c.in_channels * 2);
  L.total = o;
  return L;
}

inline uint8_t* at(void* ws, size_t off) { return reinterpret_cast<uint8_t*>(ws) + off; }
inline bf16* bat(void* ws, size_t off) { return reinterpret_cast<bf16*>(at(ws, off)); }
inline DeviceStatus* status_of(void* ws) { return reinterpret_cast<DeviceStatus*>(ws); }

inline dit_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DIT_OK : DIT_ERR_CUDA; }

#define DIT_TRY(expr)                     \
  do {                                    \
    const dit_status st_ = (expr);        \
    if (st_ != DIT_OK) return st_;        \
  } while (0)
#define DIT_CUDA(expr) DIT_TRY(cuda_status(expr))

dit_status check_stream_weights(const dit_stream_weights& w) {
  if (!aligned16(w.qkv) || !aligned16(w.q_norm) || !aligned16(w.k_norm) || !aligned16(w.out) ||
      !aligned16(w.mlp_in) || !aligned16(w.mlp_out))
    return DIT_ERR_INVALID_ARG;
  return DIT_OK;
}

// e4m3 copies: a matrix is absent (q NULL) or both pointers are 16-byte aligned; the fused
// single-stream projection is always present; a dual-block projection is given for both
// streams or for neither.
inline bool fp8_matrix_ok(const dit_fp8_matrix& m) { return !m.q || (aligned16(m.q) && aligned16(m.scale)); }

dit_status check_single_fp8(const dit_config& c, const dit_single_fp8& f) {
  if (!aligned16(f.qkv_mlp_q) || !aligned16(f.qkv_mlp_scale) || !fp8_matrix_ok(f.out)) return DIT_ERR_INVALID_ARG;
  if (f.out.q && !quantize_act_supports(c.hidden + c.mlp_hidden)) return DIT_ERR_UNSUPPORTED;
  return DIT_OK;
}

dit_status check_dual_fp8(const dit_config& c, const dit_dual_fp8& f) {
  const dit_fp8_matrix* img[4] = {&f.img.qkv, &f.img.mlp_in, &f.img.out, &f.img.mlp_out};
  const dit_fp8_matrix* txt[4] = {&f.txt.qkv, &f.txt.mlp_in, &f.txt.out, &f.txt.mlp_out};
  for (int i = 0; i < 4; ++i)
    if (!fp8_matrix_ok(*img[i]) || !fp8_matrix_ok(*txt[i]) || (img[i]->q == nullptr) != (txt[i]->q == nullptr))
      return DIT_ERR_INVALID_ARG;
  if ((f.img.out.q || f.img.mlp_out.q) && !quantize_act_supports(c.hidden + c.mlp_hidden)) return DIT_ERR_UNSUPPORTED;
  return DIT_OK;
}

dit_status check_block_args(const dit_weights* w, const dit_shape* shape, const void* x, const void* mod,
                            const float* rope, void* ws, size_t ws_bytes) {
  if (!w) return DIT_ERR_INVALID_ARG;
  DIT_TRY(check_config(&w->cfg));
  DIT_TRY(check_shape(shape));
  if (!aligned16(x) || !aligned16(mod) || !aligned16(rope) || !aligned16(ws)) return DIT_ERR_INVALID_ARG;
  if (ws_bytes < layout(w->cfg, *shape).block_end) return DIT_ERR_WORKSPACE;
  return DIT_OK;
}

// Modulation slot offsets (in units of H): img-dual 0..5, txt-dual 6..11, single 12..14,
// final 15..16.
enum { kImg = 0, kTxt = 6, kSingle = 12, kFinal = 15 };
enum { kShiftA = 0, kScaleA = 1, kGateA = 2, kShiftM = 3, kScaleM = 4, kGateM = 5 };

GemmProblemHost blank_problem() {
  GemmProblemHost p;
  memset(&p, 0, sizeof(p));
  return p;
}

dit_status run_dual_block(const dit_weights* w, int layer, const dit_shape* s, bf16* x, const bf16* mod,
                          const float* rope, void* ws, cudaStream_t st) {
  const dit_config& c = w->cfg;
  const dit_dual_weights& dw = w->dual[layer];
  const int B = s->batch, N = s->n_txt + s->n_img + s->n_ref, H = c.hidden, F = c.mlp_hidden;
  const int n_txt = s->n_txt, n_imgref = N - n_txt;
  const Layout L = layout(c, *s);
  bf16 *y = bat(ws, L.y), *q = bat(ws, L.q), *k = bat(ws, L.k), *v = bat(ws, L.v), *cat = bat(ws, L.cat);
  float* x1 = reinterpret_cast<float*>(at(ws, L.x1));  // fp32 residual stream between the two halves
  DeviceStatus* dst = status_of(ws);
  const long long ms = 17LL * H;
  auto slot = [&](int base, int which) { return mod + (long long)(base + which) * H; };
  // e4m3 projections (per kind, both streams or neither): inputs quantised per token row,
  // by the adaLN kernel (QKV, MLP-in) or by a quantising pass over cat (out, MLP-out)
  const dit_dual_fp8* f8 = w->dual_fp8 ? &w->dual_fp8[layer] : nullptr;
  const dit_stream_fp8* sf[2] = {f8 ? &f8->txt : nullptr, f8 ? &f8->img : nullptr};  // order of sw below
  const bool q_qkv = f8 && f8->img.qkv.q, q_in = f8 && f8->img.mlp_in.q;
  const bool q_out = f8 && f8->img.out.q, q_mo = f8 && f8->img.mlp_out.q;
  uint8_t* yq = at(ws, L.yq);
  float* ascale = reinterpret_cast<float*>(at(ws, L.ascale));
  uint8_t* cq = at(ws, L.cq);
  float* cscale = reinterpret_cast<float*>(at(ws, L.cscale));
  auto use_fp8 = [](GemmProblemHost& pp, const dit_fp8_matrix& m, const uint8_t* a8, const float* as, int lda) {
    pp.fp8 = 1;
    pp.a = reinterpret_cast<const bf16*>(a8);
    pp.lda = lda;
    pp.a_scale = as;
    pp.w = reinterpret_cast<const bf16*>(m.q);
    pp.w_scale = m.scale;
  };

  // 1. y = adaLN(x) with each stream's attention shift / scale
  AdaLNArgs a1{B, N, H, x, 0, (long long)N * H, 0, y, (long long)N * H, n_txt,
               slot(kTxt, kShiftA), slot(kTxt, kScaleA), slot(kImg, kShiftA), slot(kImg, kScaleA), ms, c.eps};
  if (q_qkv) {
    a1.y_q = yq;
    a1.y_scale = ascale;
  }
  a1.status = dst;
  DIT_CUDA(launch_adaln(a1, st));

  // 2. per-stream QKV projection + QK-RMSNorm + RoPE, head-major Q/K/V
  GemmProblemHost p[2];
  const dit_stream_weights* sw[2] = {&dw.txt, &dw.img};
  const int row0[2] = {0, n_txt}, rows[2] = {n_txt, n_imgref};
  for (int i = 0; i < 2; ++i) {
    p[i] = blank_problem();
    p[i].a = y; p[i].a_rows_total = N; p[i].lda = H; p[i].a_row0 = row0[i]; p[i].rows = rows[i];
    p[i].w = (const bf16*)sw[i]->qkv; p[i].n = 3 * H; p[i].k = H; p[i].epi = kEpiQKV;
    p[i].n_qkv = 3 * H; p[i].hidden = H; p[i].q = q; p[i].kk = k; p[i].v = v;
    p[i].q_norm = (const bf16*)sw[i]->q_norm; p[i].k_norm = (const bf16*)sw[i]->k_norm;
    p[i].rope = rope; p[i].seq = N; p[i].tok0 = row0[i];
    if (q_qkv) use_fp8(p[i], sf[i]->qkv, yq, ascale, H);
  }
  DIT_CUDA(launch_gemm(p, 2, B, c.eps, dst, kClsGemmQKV, st));

  // 3. joint attention over all N rows -> cat[:, :, 0:H]
  DIT_CUDA(launch_attention(B, c.heads, N, q, k, v, cat, H + F, dst, st));

  // 4. x1 = x + gate_a * (attn out^T), per stream; x1 kept in fp32 so the block rounds
  //    the residual stream to bf16 once
  const int gate_a[2] = {kTxt + kGateA, kImg + kGateA};
  if (q_out) DIT_CUDA(launch_quantize_act(cat, (long long)N * (H + F), H + F, 0, B, N, H, cq, cscale, st));
  for (int i = 0; i < 2; ++i) {
    p[i] = blank_problem();
    p[i].a = cat; p[i].a_rows_total = N; p[i].lda = H + F; p[i].a_row0 = row0[i]; p[i].rows = rows[i];
    p[i].w = (const bf16*)sw[i]->out; p[i].n = H; p[i].k = H; p[i].epi = kEpiResidual;
    p[i].res = x; p[i].out_f32 = x1; p[i].out_bstride = (long long)N * H; p[i].ld_out = H; p[i].out_row0 = row0[i];
    p[i].gate = mod + (long long)gate_a[i] * H; p[i].gate_stride = ms;
    if (q_out) use_fp8(p[i], sf[i]->out, cq, cscale, H);
  }
  DIT_CUDA(launch_gemm(p, 2, B, c.eps, dst, kClsGemmDualOut, st));

  // 5. y = adaLN(x1) with each stream's MLP shift / scale
  AdaLNArgs a2{B, N, H, x1, 1, (long long)N * H, 0, y, (long long)N * H, n_txt,
               slot(kTxt, kShiftM), slot(kTxt, kScaleM), slot(kImg, kShiftM), slot(kImg, kScaleM), ms, c.eps};
  if (q_in) {
    a2.y_q = yq;
    a2.y_scale = ascale;
  }
  a2.status = dst;
  DIT_CUDA(launch_adaln(a2, st));

  // 6. act = silu(y Wg^T) * (y Wu^T) -> cat[:, :, H:H+F], per stream
  for (int i = 0; i < 2; ++i) {
    p[i] = blank_problem();
    p[i].a = y; p[i].a_rows_total = N; p[i].lda = H; p[i].a_row0 = row0[i]; p[i].rows = rows[i];
    p[i].w = (const bf16*)sw[i]->mlp_in; p[i].n = 2 * F; p[i].k = H; p[i].epi = kEpiSwiGLU;
    p[i].out = cat; p[i].out_bstride = (long long)N * (H + F); p[i].ld_out = H + F; p[i].out_row0 = row0[i];
    p[i].out_col0 = H;
    if (q_in) use_fp8(p[i], sf[i]->mlp_in, yq, ascale, H);
  }
  DIT_CUDA(launch_gemm(p, 2, B, c.eps, dst, kClsGemmSwiGLU, st));

  // 7. x = x1 + gate_m * (act mlp_out^T), per stream
  const int gate_m[2] = {kTxt + kGateM, kImg + kGateM};
  if (q_mo) DIT_CUDA(launch_quantize_act(cat, (long long)N * (H + F), H + F, H, B, N, F, cq, cscale, st));
  for (int i = 0; i < 2; ++i) {
    p[i] = blank_problem();
    p[i].a = cat + H; p[i].a_rows_total = N; p[i].lda = H + F; p[i].a_row0 = row0[i]; p[i].rows = rows[i];
    p[i].w = (const bf16*)sw[i]->mlp_out; p[i].n = H; p[i].k = F; p[i].epi = kEpiResidual;
    p[i].res_f32 = x1; p[i].out = x; p[i].out_bstride = (long long)N * H; p[i].ld_out = H; p[i].out_row0 = row0[i];
    p[i].gate = mod + (long long)gate_m[i] * H; p[i].gate_stride = ms;
    if (q_mo) use_fp8(p[i], sf[i]->mlp_out, cq, cscale, F);
  }
  DIT_CUDA(launch_gemm(p, 2, B, c.eps, dst, kClsGemmDualMlpOut, st));
  return DIT_OK;
}

dit_status run_single_block(const dit_weights* w, int layer, const dit_shape* s, bf16* x, const bf16* mod,
                            const float* rope, void* ws, cudaStream_t st) {
  const dit_config& c = w->cfg;
  const dit_single_weights& sw = w->single[layer];
  const int B = s->batch, N = s->n_txt + s->n_img + s->n_ref, H = c.hidden, F = c.mlp_hidden;
  const Layout L = layout(c, *s);
  bf16 *y = bat(ws, L.y), *q = bat(ws, L.q), *k = bat(ws, L.k), *v = bat(ws, L.v), *cat = bat(ws, L.cat);
  DeviceStatus* dst = status_of(ws);
  const long long ms = 17LL * H;
  const bf16* sh = mod + (long long)(kSingle + 0) * H;
  const bf16* sc = mod + (long long)(kSingle + 1) * H;

  const dit_single_fp8* f8 = w->single_fp8 ? &w->single_fp8[layer] : nullptr;
  AdaLNArgs a1{B, N, H, x, 0, (long long)N * H, 0, y, (long long)N * H, 0, sh, sc, sh, sc, ms, c.eps};
  if (f8) {
    a1.y_q = at(ws, L.yq);
    a1.y_scale = reinterpret_cast<float*>(at(ws, L.ascale));
  }
  a1.status = dst;
  DIT_CUDA(launch_adaln(a1, st));

  GemmProblemHost p = blank_problem();
  p.a = f8 ? reinterpret_cast<const bf16*>(at(ws, L.yq)) : y;
  p.a_rows_total = N; p.lda = H; p.a_row0 = 0; p.rows = N;
  p.w = f8 ? (const bf16*)f8->qkv_mlp_q : (const bf16*)sw.qkv_mlp; p.n = 3 * H + 2 * F; p.k = H; p.epi = kEpiQKV;
  if (f8) {
    p.fp8 = 1;
    p.a_scale = reinterpret_cast<const float*>(at(ws, L.ascale));
    p.w_scale = f8->qkv_mlp_scale;
  }
  p.n_qkv = 3 * H; p.hidden = H; p.q = q; p.kk = k; p.v = v;
  p.q_norm = (const bf16*)sw.q_norm; p.k_norm = (const bf16*)sw.k_norm; p.rope = rope; p.seq = N; p.tok0 = 0;
  p.out = cat; p.out_bstride = (long long)N * (H + F); p.ld_out = H + F; p.out_row0 = 0; p.out_col0 = H;
  DIT_CUDA(launch_gemm(&p, 1, B, c.eps, dst, kClsGemmFused, st));

  DIT_CUDA(launch_attention(B, c.heads, N, q, k, v, cat, H + F, dst, st));

  p = blank_problem();
  p.a = cat; p.a_rows_total = N; p.lda = H + F; p.a_row0 = 0; p.rows = N;
  p.w = (const bf16*)sw.out; p.n = H; p.k = H + F; p.epi = kEpiResidual;
  p.out = x; p.out_bstride = (long long)N * H; p.ld_out = H; p.out_row0 = 0;
  p.gate = mod + (long long)(kSingle + 2) * H; p.gate_stride = ms;
  if (f8 && f8->out.q) {
    // e4m3 out-projection: [attn | act] quantised per token row first
    uint8_t* cq = at(ws, L.cq);
    float* cscale = reinterpret_cast<float*>(at(ws, L.cscale));
    DIT_CUDA(launch_quantize_act(cat, (long long)N * (H + F), H + F, 0, B, N, H + F, cq, cscale, st));
    p.fp8 = 1;
    p.a = reinterpret_cast<const bf16*>(cq);
    p.a_scale = cscale;
    p.w = reinterpret_cast<const bf16*>(f8->out.q);
    p.w_scale = f8->out.scale;
  }
  DIT_CUDA(launch_gemm(&p, 1, B, c.eps, dst, kClsGemmSingleOut, st));
  return DIT_OK;
}

dit_status run_modulation_into(const dit_weights* w, const float* sigma, int batch, bf16* mod, float* h1, float* h2,
                               cudaStream_t st) {
  const int H = w->cfg.hidden;
  DIT_CUDA(launch_timestep_in((const bf16*)w->mod.t_in, H, 256, sigma, batch, h1, st));
  DIT_CUDA(launch_gemv((const bf16*)w->mod.t_out, H, H, h1, batch, 1, h2, nullptr, st));
  DIT_CUDA(launch_gemv((const bf16*)w->mod.mod, 17 * H, H, h2, batch, 0, nullptr, mod, st));
  return DIT_OK;
}

dit_status run_modulation(const dit_weights* w, const float* sigma, int batch, bf16* mod, void* ws,
                          const Layout& L, cudaStream_t st) {
  const int H = w->cfg.hidden;
  float* h1 = reinterpret_cast<float*>(at(ws, L.h1));
  float* h2 = reinterpret_cast<float*>(at(ws, L.h2));
  DIT_CUDA(launch_timestep_in((const bf16*)w->mod.t_in, H, 256, sigma, batch, h1, st));
  DIT_CUDA(launch_gemv((const bf16*)w->mod.t_out, H, H, h1, batch, 1, h2, nullptr, st));
  DIT_CUDA(launch_gemv((const bf16*)w->mod.mod, 17 * H, H, h2, batch, 0, nullptr, mod, st));
  return DIT_OK;
}

dit_status check_step_weights(const dit_weights* w) {
  if (!w) return DIT_ERR_INVALID_ARG;
  DIT_TRY(check_config(&w->cfg));
  if (!aligned16(w->mod.t_in) || !aligned16(w->mod.t_out) || !aligned16(w->mod.mod) || !aligned16(w->x_emb) ||
      !aligned16(w->ctx_emb) || !aligned16(w->proj_out))
    return DIT_ERR_INVALID_ARG;
  if (w->cfg.n_dual > 0 && !w->dual) return DIT_ERR_INVALID_ARG;
  if (w->cfg.n_single > 0 && !w->single) return DIT_ERR_INVALID_ARG;
  for (int i = 0; i < w->cfg.n_dual; ++i) {
    DIT_TRY(check_stream_weights(w->dual[i].img));
    DIT_TRY(check_stream_weights(w->dual[i].txt));
    if (w->dual_fp8) DIT_TRY(check_dual_fp8(w->cfg, w->dual_fp8[i]));
  }
  for (int i = 0; i < w->cfg.n_single; ++i) {
    const dit_single_weights& s = w->single[i];
    if (!aligned16(s.qkv_mlp) || !aligned16(s.q_norm) || !aligned16(s.k_norm) || !aligned16(s.out))
      return DIT_ERR_INVALID_ARG;
    if (w->single_fp8) DIT_TRY(check_single_fp8(w->cfg, w->single_fp8[i]));
  }
  return DIT_OK;
}

// Where the final projection writes: the velocity (STORE), or, in the denoising loop, the
// Euler update x_next = x + coef_b * v into an fp32 state and a bf16 copy.
struct FinalOut {
  bf16* vel;
  const bf16* res_bf;
  const float* res_f32;
  const float* coef;
  float* state;
  bf16* out_bf;
};

dit_status run_step_core(const dit_weights* w, const dit_shape* s, const bf16* img, const bf16* ref,
                         const bf16* txt, const float* rope, const bf16* mod, const FinalOut& fin, void* ws,
                         cudaStream_t st) {
  const dit_config& c = w->cfg;
  const Layout L = layout(c, *s);
  const int B = s->batch, N = s->n_txt + s->n_img + s->n_ref, H = c.hidden, C = c.in_channels;
  bf16* x = bat(ws, L.x);
  bf16* y = bat(ws, L.y);
  DeviceStatus* dst = status_of(ws);

  // Embedders: text rows by ctx_emb, target-image rows by x_emb, into one [B, N, H].
  GemmProblemHost p[2];
  p[0] = blank_problem();
  p[0].a = txt; p[0].a_rows_total = s->n_txt; p[0].lda = c.txt_dim; p[0].rows = s->n_txt;
  p[0].w = (const bf16*)w->ctx_emb; p[0].n = H; p[0].k = c.txt_dim; p[0].epi = kEpiStore;
  p[0].out = x; p[0].out_bstride = (long long)N * H; p[0].ld_out = H; p[0].out_row0 = 0;
  p[1] = blank_problem();
  p[1].a = img; p[1].a_rows_total = s->n_img; p[1].lda = C; p[1].rows = s->n_img;
  p[1].w = (const bf16*)w->x_emb; p[1].n = H; p[1].k = C; p[1].epi = kEpiStore;
  p[1].out = x; p[1].out_bstride = (long long)N * H; p[1].ld_out = H; p[1].out_row0 = s->n_txt;
  DIT_CUDA(launch_gemm(p, 2, B, c.eps, dst, kClsGemmPlain, st));
  if (s->n_ref > 0) {
    p[0] = blank_problem();
    p[0].a = ref; p[0].a_rows_total = s->n_ref; p[0].lda = C; p[0].rows = s->n_ref;
    p[0].w = (const bf16*)w->x_emb; p[0].n = H; p[0].k = C; p[0].epi = kEpiStore;
    p[0].out = x; p[0].out_bstride = (long long)N * H; p[0].ld_out = H; p[0].out_row0 = s->n_txt + s->n_img;
    DIT_CUDA(launch_gemm(p, 1, B, c.eps, dst, kClsGemmPlain, st));
  }

  for (int i = 0; i < c.n_dual; ++i) DIT_TRY(run_dual_block(w, i, s, x, mod, rope, ws, st));
  for (int i = 0; i < c.n_single; ++i) DIT_TRY(run_single_block(w, i, s, x, mod, rope, ws, st));

  // Final layer on the target-image rows only.
  const long long ms = 17LL * H;
  const bf16* fsh = mod + (long long)(kFinal + 0) * H;
  const bf16* fsc = mod + (long long)(kFinal + 1) * H;
  AdaLNArgs af{B, s->n_img, H, x, 0, (long long)N * H, s->n_txt, y, (long long)s->n_img * H, 0, fsh, fsc, fsh, fsc, ms,
               c.eps};
  af.status = status_of(ws);
  DIT_CUDA(launch_adaln(af, st));
  p[0] = blank_problem();
  p[0].a = y; p[0].a_rows_total = s->n_img; p[0].lda = H; p[0].rows = s->n_img;
  p[0].w = (const bf16*)w->proj_out; p[0].n = C; p[0].k = H;
  p[0].out_bstride = (long long)s->n_img * C; p[0].ld_out = C; p[0].out_row0 = 0;
  if (fin.vel) {
    p[0].epi = kEpiStore;
    p[0].out = fin.vel;
  } else {
    p[0].epi = kEpiResidual;
    p[0].res = fin.res_bf;
    p[0].res_f32 = fin.res_f32;
    p[0].coef = fin.coef;
    p[0].out_f32 = fin.state;
    p[0].out = fin.out_bf;
  }
  DIT_CUDA(launch_gemm(p, 1, B, c.eps, dst, kClsGemmPlain, st));
  return DIT_OK;
}

dit_status run_step(const dit_weights* w, const dit_shape* s, const bf16* img, const bf16* ref, const bf16* txt,
                    const float* rope, const float* sigma, bf16* vel, void* ws, cudaStream_t st) {
  const Layout L = layout(w->cfg, *s);
  bf16* mod = bat(ws, L.mod);
  DIT_TRY(run_modulation(w, sigma, s->batch, mod, ws, L, st));
  FinalOut fin{vel, nullptr, nullptr, nullptr, nullptr, nullptr};
  return run_step_core(w, s, img, ref, txt, rope, mod, fin, ws, st);
}

}  // namespace
}  // namespace dit

using namespace dit;

// ---------------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------------
extern "C" {

const char* dit_status_string(dit_status s) {
  switch (s) {
    case DIT_OK: return "ok";
    case DIT_ERR_INVALID_ARG: return "invalid argument";
    case DIT_ERR_UNSUPPORTED: return "unsupported configuration";
    case DIT_ERR_WORKSPACE: return "workspace too small";
    case DIT_ERR_CUDA: return "CUDA error";
    case DIT_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

dit_status dit_config_klein(dit_config* cfg) {
  if (!cfg) return DIT_ERR_INVALID_ARG;
  cfg->hidden = 3072;
  cfg->heads = 24;
  cfg->head_dim = 128;
  cfg->mlp_hidden = 9216;
  cfg->n_dual = 5;
  cfg->n_single = 20;
  cfg->in_channels = 128;
  cfg->txt_dim = 7680;
  cfg->rope_theta = 2000.0f;
  for (int i = 0; i < 4; ++i) cfg->axes_dim[i] = 32;
  cfg->eps = 1e-6f;
  return DIT_OK;
}

dit_status dit_workspace_size(const dit_config* cfg, const dit_shape* shape, size_t* bytes) {
  DIT_TRY(check_config(cfg));
  DIT_TRY(check_shape(shape));
  if (!bytes) return DIT_ERR_INVALID_ARG;
  *bytes = layout(*cfg, *shape).total;
  return DIT_OK;
}

dit_status dit_token_ids(const dit_shape* shape, int grid_h, int grid_w, const int* ref_grids_host, int n_refs,
                         int32_t* ids_host) {
  DIT_TRY(check_shape(shape));
  if (!ids_host || grid_h < 1 || grid_w < 1 || n_refs < 0 || (n_refs > 0 && !ref_grids_host))
    return DIT_ERR_INVALID_ARG;
  if ((long long)grid_h * grid_w != shape->n_img) return DIT_ERR_INVALID_ARG;
  long long nref = 0;
  for (int i = 0; i < n_refs; ++i) {
    if (ref_grids_host[2 * i] < 1 || ref_grids_host[2 * i + 1] < 1) return DIT_ERR_INVALID_ARG;
    nref += (long long)ref_grids_host[2 * i] * ref_grids_host[2 * i + 1];
    if (nref > shape->n_ref) return DIT_ERR_INVALID_ARG;  // also keeps the sum far from overflow
  }
  if (nref != shape->n_ref) return DIT_ERR_INVALID_ARG;
  int32_t* o = ids_host;
  auto put = [&](int t, int h, int w, int l) {
    o[0] = t;
    o[1] = h;
    o[2] = w;
    o[3] = l;
    o += 4;
  };
  for (int i = 0; i < shape->n_txt; ++i) put(0, 0, 0, i);
  for (int r = 0; r < grid_h; ++r)
    for (int c = 0; c < grid_w; ++c) put(0, r, c, 0);
  for (int i = 0; i < n_refs; ++i)
    for (int r = 0; r < ref_grids_host[2 * i]; ++r)
      for (int c = 0; c < ref_grids_host[2 * i + 1]; ++c) put(10 + 10 * i, r, c, 0);
  return DIT_OK;
}

dit_status dit_rope_table(const dit_config* cfg, const int32_t* ids_dev, int n, float* table_dev,
                          dit_stream_t stream) {
  DIT_TRY(check_config(cfg));
  if (n < 0 || n > kMaxTokens) return DIT_ERR_INVALID_ARG;
  if (n == 0) return DIT_OK;
  if (!aligned16(ids_dev) || !aligned16(table_dev)) return DIT_ERR_INVALID_ARG;
  return cuda_status(launch_rope_table(ids_dev, n, cfg->axes_dim, cfg->rope_theta, table_dev, (cudaStream_t)stream));
}

dit_status dit_pack_mlp_in(const void* src_dev, void* dst_dev, int mlp_hidden, int cols, dit_stream_t stream) {
  if (!aligned16(src_dev) || !aligned16(dst_dev)) return DIT_ERR_INVALID_ARG;
  if (mlp_hidden <= 0 || mlp_hidden % 128 != 0 || mlp_hidden > kMaxTokens / 2 || cols <= 0 || cols % 8 != 0 ||
      cols > kMaxTokens)
    return DIT_ERR_INVALID_ARG;
  const uintptr_t a = (uintptr_t)src_dev, b = (uintptr_t)dst_dev, len = (uintptr_t)2 * mlp_hidden * cols * 2;
  if (a < b + len && b < a + len) return DIT_ERR_INVALID_ARG;
  return cuda_status(launch_pack_mlp_in((const bf16*)src_dev, (bf16*)dst_dev, mlp_hidden, cols, (cudaStream_t)stream));
}

dit_status dit_quantize_rows_fp8(const void* w_dev, int rows, int cols, void* q_dev, float* scale_dev,
                                 dit_stream_t stream) {
  if (!aligned16(w_dev) || !aligned16(q_dev) || !aligned16(scale_dev) || rows < 1 || rows > kMaxTokens || cols < 16 ||
      cols % 16 != 0 || cols > kMaxTokens)
    return DIT_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_rows((const bf16*)w_dev, rows, cols, (uint8_t*)q_dev, scale_dev,
                                          (cudaStream_t)stream));
}

dit_status dit_modulation(const dit_weights* w, const float* sigma_dev, int batch, void* mod_dev, void* ws,
                          size_t ws_bytes, dit_stream_t stream) {
  if (!w) return DIT_ERR_INVALID_ARG;
  DIT_TRY(check_config(&w->cfg));
  if (batch < 1 || batch > kMaxBatch) return DIT_ERR_INVALID_ARG;
  if (!aligned16(w->mod.t_in) || !aligned16(w->mod.t_out) || !aligned16(w->mod.mod)) return DIT_ERR_INVALID_ARG;
  if (!aligned16(sigma_dev) || !aligned16(mod_dev) || !aligned16(ws)) return DIT_ERR_INVALID_ARG;
  const dit_shape s{batch, 1, 1, 0};
  const Layout L = layout(w->cfg, s);
  if (ws_bytes < L.h2 + (size_t)batch * w->cfg.hidden * 4) return DIT_ERR_WORKSPACE;
  return run_modulation(w, sigma_dev, batch, (bf16*)mod_dev, ws, L, (cudaStream_t)stream);
}

dit_status dit_dual_block_fwd(const dit_weights* w, int layer, const dit_shape* shape, void* x_dev,
                              const void* mod_dev, const float* rope_dev, void* ws, size_t ws_bytes,
                              dit_stream_t stream) {
  DIT_TRY(check_block_args(w, shape, x_dev, mod_dev, rope_dev, ws, ws_bytes));
  if (layer < 0 || layer >= w->cfg.n_dual || !w->dual) return DIT_ERR_INVALID_ARG;
  DIT_TRY(check_stream_weights(w->dual[layer].img));
  DIT_TRY(check_stream_weights(w->dual[layer].txt));
  if (w->dual_fp8) DIT_TRY(check_dual_fp8(w->cfg, w->dual_fp8[layer]));
  return run_dual_block(w, layer, shape, (bf16*)x_dev, (const bf16*)mod_dev, rope_dev, ws, (cudaStream_t)stream);
}

dit_status dit_single_block_fwd(const dit_weights* w, int layer, const dit_shape* shape, void* x_dev,
                                const void* mod_dev, const float* rope_dev, void* ws, size_t ws_bytes,
                                dit_stream_t stream) {
  DIT_TRY(check_block_args(w, shape, x_dev, mod_dev, rope_dev, ws, ws_bytes));
  if (layer < 0 || layer >= w->cfg.n_single || !w->single) return DIT_ERR_INVALID_ARG;
  const dit_single_weights& s = w->single[layer];
  if (!aligned16(s.qkv_mlp) || !aligned16(s.q_norm) || !aligned16(s.k_norm) || !aligned16(s.out))
    return DIT_ERR_INVALID_ARG;
  if (w->single_fp8) DIT_TRY(check_single_fp8(w->cfg, w->single_fp8[layer]));
  return run_single_block(w, layer, shape, (bf16*)x_dev, (const bf16*)mod_dev, rope_dev, ws, (cudaStream_t)stream);
}

dit_status dit_step_fwd(const dit_weights* w, const dit_shape* shape, const void* img_tokens,
                        const void* ref_tokens, const void* txt_emb, const float* rope_dev, const float* sigma_dev,
                        void* velocity_out, void* ws, size_t ws_bytes, dit_stream_t stream) {
  DIT_TRY(check_step_weights(w));
  DIT_TRY(check_shape(shape));
  if (!aligned16(img_tokens) || !aligned16(txt_emb) || !aligned16(rope_dev) || !aligned16(sigma_dev) ||
      !aligned16(velocity_out) || !aligned16(ws))
    return DIT_ERR_INVALID_ARG;
  if ((shape->n_ref > 0) != (ref_tokens != nullptr)) return DIT_ERR_INVALID_ARG;
  if (ref_tokens && !aligned16(ref_tokens)) return DIT_ERR_INVALID_ARG;
  if (ws_bytes < layout(w->cfg, *shape).step_end) return DIT_ERR_WORKSPACE;
  return run_step(w, shape, (const bf16*)img_tokens, (const bf16*)ref_tokens, (const bf16*)txt_emb, rope_dev,
                  sigma_dev, (bf16*)velocity_out, ws, (cudaStream_t)stream);
}

dit_status dit_denoise_fwd(const dit_weights* w, const dit_shape* shape, void* x_tokens, const void* ref_tokens,
                           const void* txt_emb, const float* rope_dev, const float* sigmas_host, int steps, void* ws,
                           size_t ws_bytes, dit_stream_t stream) {
  DIT_TRY(check_step_weights(w));
  DIT_TRY(check_shape(shape));
  if (!aligned16(x_tokens) || !aligned16(txt_emb) || !aligned16(rope_dev) || !aligned16(ws) || !sigmas_host)
    return DIT_ERR_INVALID_ARG;
  if ((shape->n_ref > 0) != (ref_tokens != nullptr)) return DIT_ERR_INVALID_ARG;
  if (ref_tokens && !aligned16(ref_tokens)) return DIT_ERR_INVALID_ARG;
  if (steps < 1 || steps > kMaxDenoiseSteps) return DIT_ERR_INVALID_ARG;
  for (int k = 0; k <= steps; ++k)
    if (!(sigmas_host[k] >= 0.f && sigmas_host[k] <= 1000.f)) return DIT_ERR_INVALID_ARG;
  const Layout L = layout(w->cfg, *shape);
  if (ws_bytes < L.total) return DIT_ERR_WORKSPACE;
  const cudaStream_t st = (cudaStream_t)stream;
  const int B = shape->batch, H = w->cfg.hidden;
  float* sig = reinterpret_cast<float*>(at(ws, L.den_sigma));
  float* coef = reinterpret_cast<float*>(at(ws, L.den_coef));
  bf16* mod = bat(ws, L.den_mod);
  DIT_CUDA(launch_denoise_setup(sigmas_host, steps, B, sig, coef, st));
  // The modulation of every step at once: rows k*B + b, at most 8 rows per weight pass.
  const int rows = steps * B;
  for (int r0 = 0; r0 < rows; r0 += 8) {
    const int nr = rows - r0 < 8 ? rows - r0 : 8;
    DIT_TRY(run_modulation_into(w, sig + r0, nr, mod + (long long)r0 * 17 * H,
                                reinterpret_cast<float*>(at(ws, L.den_h1)), reinterpret_cast<float*>(at(ws, L.den_h2)),
                                st));
  }
  bf16* xt = (bf16*)x_tokens;
  bf16* xbf = bat(ws, L.den_xbf);
  float* state = reinterpret_cast<float*>(at(ws, L.den_state));
  for (int k = 0; k < steps; ++k) {
    const bool first = k == 0, last = k == steps - 1;
    FinalOut fin{nullptr, first ? xt : nullptr, first ? nullptr : state, coef + (long long)k * B, state,
                 last ? xt : xbf};
    DIT_TRY(run_step_core(w, shape, first ? xt : xbf, (const bf16*)ref_tokens, (const bf16*)txt_emb, rope_dev,
                          mod + (long long)k * B * 17 * H, fin, ws, st));
  }
  return DIT_OK;
}

dit_status dit_step_host(const dit_weights* w, const dit_shape* shape, const void* img_tokens_host,
                         const void* ref_tokens_host, const void* txt_emb_host, const float* rope_dev,
                         const float* sigma_host, void* velocity_host, void* ws, size_t ws_bytes,
                         dit_stream_t stream) {
  DIT_TRY(check_step_weights(w));
  DIT_TRY(check_shape(shape));
  if (!img_tokens_host || !txt_emb_host || !sigma_host || !velocity_host || !aligned16(rope_dev) || !aligned16(ws))
    return DIT_ERR_INVALID_ARG;
  if ((shape->n_ref > 0) != (ref_tokens_host != nullptr)) return DIT_ERR_INVALID_ARG;
  const Layout L = layout(w->cfg, *shape);
  if (ws_bytes < L.total) return DIT_ERR_WORKSPACE;
  const cudaStream_t st = (cudaStream_t)stream;
  const size_t B = shape->batch, C = w->cfg.in_channels;
  const size_t img_b = B * shape->n_img * C * 2, ref_b = B * shape->n_ref * C * 2,
               txt_b = B * shape->n_txt * (size_t)w->cfg.txt_dim * 2;
  DIT_CUDA(cudaMemcpyAsync(at(ws, L.in_img), img_tokens_host, img_b, cudaMemcpyHostToDevice, st));
  if (ref_b) DIT_CUDA(cudaMemcpyAsync(at(ws, L.in_ref), ref_tokens_host, ref_b, cudaMemcpyHostToDevice, st));
  DIT_CUDA(cudaMemcpyAsync(at(ws, L.in_txt), txt_emb_host, txt_b, cudaMemcpyHostToDevice, st));
  DIT_CUDA(cudaMemcpyAsync(at(ws, L.in_sigma), sigma_host, B * 4, cudaMemcpyHostToDevice, st));
  DIT_TRY(run_step(w, shape, bat(ws, L.in_img), ref_b ? bat(ws, L.in_ref) : nullptr, bat(ws, L.in_txt), rope_dev,
                   reinterpret_cast<const float*>(at(ws, L.in_sigma)), bat(ws, L.out_vel), ws, st));
  DIT_CUDA(cudaMemcpyAsync(velocity_host, at(ws, L.out_vel), img_b, cudaMemcpyDeviceToHost, st));
  return DIT_OK;
}

}  // extern "C"

struct dit_graph_s {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  unsigned long long kernels;  // kernel launches one replay performs
};

extern "C" {

dit_status dit_step_graph_create(const dit_weights* w, const dit_shape* shape, const void* img_tokens,
                                 const void* ref_tokens, const void* txt_emb, const float* rope_dev,
                                 const float* sigma, void* velocity_out, void* ws, size_t ws_bytes, int host_io,
                                 dit_stream_t stream, dit_graph* graph_out) {
  if (!graph_out) return DIT_ERR_INVALID_ARG;
  *graph_out = nullptr;
  const cudaStream_t st = (cudaStream_t)stream;
  auto enqueue = [&](dit_stream_t on) -> dit_status {
    return host_io ? dit_step_host(w, shape, img_tokens, ref_tokens, txt_emb, rope_dev, sigma, velocity_out, ws,
                                   ws_bytes, on)
                   : dit_step_fwd(w, shape, img_tokens, ref_tokens, txt_emb, rope_dev, sigma, velocity_out, ws,
                                  ws_bytes, on);
  };
  // Warm-up: validates every argument and performs the one-time per-kernel set-up
  // (shared-memory attributes) outside the capture.
  DIT_TRY(enqueue(stream));
  DIT_CUDA(cudaStreamSynchronize(st));
  // Capture on a private stream: the caller's may be the legacy default stream, which
  // cannot be captured.  The graph is replayed on any stream later.
  cudaStream_t cap = nullptr;
  DIT_CUDA(cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking));
  cudaGraph_t g = nullptr;
  cudaError_t ce = cudaStreamBeginCapture(cap, cudaStreamCaptureModeThreadLocal);
  dit_status es = DIT_OK;
  // Captured launches do not run: count them when the graph is replayed instead.
  t_capturing = true;
  t_captured = 0;
  if (ce == cudaSuccess) {
    es = enqueue((dit_stream_t)cap);
    ce = cudaStreamEndCapture(cap, &g);
  }
  t_capturing = false;
  const unsigned long long kernels = t_captured;
  cudaStreamDestroy(cap);
  if (es != DIT_OK || ce != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();  // do not leave this failure for the next launch check to find
    return es != DIT_OK ? es : DIT_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  if (cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    cudaGetLastError();
    return DIT_ERR_CUDA;
  }
  dit_graph h = new (std::nothrow) dit_graph_s{g, exec, kernels};
  if (!h) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(g);
    return DIT_ERR_CUDA;
  }
  *graph_out = h;
  return DIT_OK;
}

dit_status dit_graph_launch(dit_graph graph, dit_stream_t stream) {
  if (!graph) return DIT_ERR_INVALID_ARG;
  g_launches.fetch_add(graph->kernels, std::memory_order_relaxed);
  return cuda_status(cudaGraphLaunch(graph->exec, (cudaStream_t)stream));
}

dit_status dit_graph_destroy(dit_graph graph) {
  if (!graph) return DIT_OK;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
  return DIT_OK;
}

dit_status dit_sync_status(void* ws, dit_stream_t stream, uint32_t* where_out) {
  if (!aligned16(ws)) return DIT_ERR_INVALID_ARG;
  const cudaStream_t st = (cudaStream_t)stream;
  DeviceStatus h;
  DIT_CUDA(cudaMemcpyAsync(&h, ws, 8, cudaMemcpyDeviceToHost, st));
  DIT_CUDA(cudaStreamSynchronize(st));
  if (where_out) *where_out = h.where;
  if (h.word != 0) {
    DIT_CUDA(cudaMemsetAsync(ws, 0, 8, st));
    DIT_CUDA(cudaStreamSynchronize(st));
    return DIT_ERR_TIMEOUT;
  }
  return DIT_OK;
}

dit_status dit_selftest_wait_timeout(void* ws, size_t ws_bytes, unsigned int limit_us, dit_stream_t stream) {
  if (!aligned16(ws) || ws_bytes < sizeof(DeviceStatus) || limit_us < 1 || limit_us > 1000000)
    return DIT_ERR_INVALID_ARG;
  return cuda_status(launch_selftest_wait(status_of(ws), 1000ull * limit_us, (cudaStream_t)stream));
}

dit_status dit_adaln(int batch, int rows, int hidden, const void* x_dev, int x_rows, int x_row0, int split,
                     const void* shift_lo, const void* scale_lo, const void* shift_hi, const void* scale_hi,
                     long long mod_stride, float eps, void* y_dev, dit_stream_t stream) {
  if (batch < 1 || batch > kMaxBatch || rows < 0 || rows > kMaxTokens || x_rows < 0 || x_row0 < 0 ||
      (long long)x_row0 + rows > x_rows)
    return DIT_ERR_INVALID_ARG;
  if (!adaln_supports(hidden)) return DIT_ERR_UNSUPPORTED;
  if (!aligned16(x_dev) || !aligned16(y_dev) || !aligned16(shift_lo) || !aligned16(scale_lo) ||
      !aligned16(shift_hi) || !aligned16(scale_hi) || mod_stride < 0 || mod_stride % 8 != 0 || !(eps > 0.f))
    return DIT_ERR_INVALID_ARG;
  AdaLNArgs a{batch, rows, hidden, x_dev, 0, (long long)x_rows * hidden, x_row0, (bf16*)y_dev,
              (long long)rows * hidden, split, (const bf16*)shift_lo, (const bf16*)scale_lo, (const bf16*)shift_hi,
              (const bf16*)scale_hi, mod_stride, eps};
  return cuda_status(launch_adaln(a, (cudaStream_t)stream));
}

dit_status dit_linear(int batch, int rows, int n_out, int k, const void* a_dev, const void* w_dev, void* out_dev,
                      int ld_out, dit_epilogue epi, const void* gate_dev, long long gate_stride, void* ws,
                      size_t ws_bytes, dit_stream_t stream) {
  // rows, n_out and k up to the token limit keep every tile count and offset of the GEMM in
  // range (tiles <= 4096 x 4096 x 64 < 2^31)
  if (batch < 1 || batch > kMaxBatch || rows < 1 || rows > kMaxTokens || n_out < 1 || n_out > kMaxTokens || k < 1 ||
      k > kMaxTokens || k % 8 != 0 || n_out % 32 != 0 || ld_out < n_out || ld_out % 8 != 0)
    return DIT_ERR_INVALID_ARG;
  if (!aligned16(a_dev) || !aligned16(w_dev) || !aligned16(out_dev) || !aligned16(ws)) return DIT_ERR_INVALID_ARG;
  if (ws_bytes < sizeof(DeviceStatus)) return DIT_ERR_WORKSPACE;
  GemmProblemHost p = blank_problem();
  p.a = (const bf16*)a_dev; p.a_rows_total = rows; p.lda = k; p.rows = rows;
  p.w = (const bf16*)w_dev; p.n = n_out; p.k = k;
  p.out = (bf16*)out_dev; p.out_bstride = (long long)rows * ld_out; p.ld_out = ld_out;
  int cls = kClsGemmPlain;
  switch (epi) {
    case DIT_EPI_STORE: p.epi = kEpiStore; break;
    case DIT_EPI_GATED_RESIDUAL:
      if (!aligned16(gate_dev) || gate_stride < 0 || gate_stride % 8 != 0) return DIT_ERR_INVALID_ARG;
      p.epi = kEpiResidual; p.gate = (const bf16*)gate_dev; p.gate_stride = gate_stride; cls = kClsGemmResidual;
      break;
    case DIT_EPI_SWIGLU:
      if (n_out % 128 != 0) return DIT_ERR_INVALID_ARG;
      p.epi = kEpiSwiGLU; p.n = 2 * n_out; cls = kClsGemmSwiGLU;
      break;
    default: return DIT_ERR_INVALID_ARG;
  }
  return cuda_status(launch_gemm(&p, 1, batch, 1e-6f, status_of(ws), cls, (cudaStream_t)stream));
}

dit_status dit_attention(int batch, int heads, int n, const void* q_dev, const void* k_dev, const void* v_dev,
                         void* out_dev, int ld_out, void* ws, size_t ws_bytes, dit_stream_t stream) {
  if (batch < 1 || batch > kMaxBatch || heads < 1 || heads > kMaxTokens / 128 || n < 1 || n > kMaxTokens ||
      ld_out < 128 * heads || ld_out % 8 != 0)
    return DIT_ERR_INVALID_ARG;
  if (!aligned16(q_dev) || !aligned16(k_dev) || !aligned16(v_dev) || !aligned16(out_dev) || !aligned16(ws))
    return DIT_ERR_INVALID_ARG;
  if (ws_bytes < sizeof(DeviceStatus)) return DIT_ERR_WORKSPACE;
  return cuda_status(launch_attention(batch, heads, n, (const bf16*)q_dev, (const bf16*)k_dev, (const bf16*)v_dev,
                                      (bf16*)out_dev, ld_out, status_of(ws), (cudaStream_t)stream));
}

unsigned long long dit_launch_count(void) { return g_launches.load(); }

dit_status dit_timing_begin(int max_records) {
  if (max_records < 1 || max_records > (1 << 20)) return DIT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_timing_mu);
  for (auto& r : g_recs) {
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  g_recs.clear();
  g_recs.resize(max_records);
  for (auto& r : g_recs) {
    r.cls = -1;
    if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.stop) != cudaSuccess) {
      g_recs.clear();
      return DIT_ERR_CUDA;
    }
  }
  g_rec_used = 0;
  g_timing_on = true;
  return DIT_OK;
}

dit_status dit_timing_end(int* n, int* classes, float* ms, int cap) {
  if (!n || cap < 0 || (cap > 0 && (!classes || !ms))) return DIT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_timing_mu);
  g_timing_on = false;
  const int used = g_rec_used < cap ? g_rec_used : cap;
  for (int i = 0; i < used; ++i) {
    if (cudaEventSynchronize(g_recs[i].stop) != cudaSuccess) return DIT_ERR_CUDA;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, g_recs[i].start, g_recs[i].stop) != cudaSuccess) return DIT_ERR_CUDA;
    classes[i] = g_recs[i].cls;
    ms[i] = t;
  }
  *n = used;
  return DIT_OK;
}

const char* dit_kernel_class_name(int cls) { return kernel_class_name(cls); }

dit_status dit_timing_select(unsigned int class_mask) {
  if (class_mask == 0u) return DIT_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_timing_mu);
  g_timing_mask = class_mask;
  return DIT_OK;
}

}  // extern "C"
