// Host-side runtime shared by the launchers: launch accounting and per-launch timing,
// TMA descriptor encoding, and the internal launcher declarations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace dit {

// Kernel classes, for timing records.
enum KernelClass : int {
  kClsAdaLN = 0,
  kClsGemmQKV = 1,         // dual-stream QKV projection (+ RMSNorm + RoPE epilogue), both streams
  kClsGemmFused = 2,       // single-stream fused QKV + MLP-in projection
  kClsGemmResidual = 3,    // gated residual from the component entry point
  kClsGemmSwiGLU = 4,      // dual-stream MLP-in with SwiGLU, both streams
  kClsGemmPlain = 5,       // embedders, final projection, plain component calls
  kClsAttention = 6,
  kClsModulation = 7,
  kClsRope = 8,
  kClsPack = 9,
  kClsGemmDualOut = 10,    // dual-stream attention out-projection + gated residual
  kClsGemmDualMlpOut = 11, // dual-stream MLP-out + gated residual
  kClsGemmSingleOut = 12,  // single-stream out-projection over [attn | act] + gated residual
  kClsQuantAct = 13,       // per-row e4m3 quantisation of an out-projection's input
  kClsCount = 14
};

const char* kernel_class_name(int cls);

// Brackets one kernel launch: counts it (or, during a graph capture on this thread, adds it
// to the graph's count) and, while timing is on, records an event pair on the launch's
// stream (captured into the graph during a capture).
class LaunchScope {
 public:
  LaunchScope(int cls, cudaStream_t stream);
  ~LaunchScope();

 private:
  void record(cudaEvent_t e);
  int slot_;
  cudaStream_t stream_;
  bool captured_;
};

// Number of SMs of the current device (cached per device).
int sm_count();

// Launch a step kernel with programmatic stream serialisation (its prologue may overlap the
// previous kernel's tail; the kernel itself calls grid_dependency_wait() before touching
// dependent memory).  DIT_NO_PDL=1 in the environment turns the attribute off.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Encode a bf16 tiled TMA descriptor with 128-byte swizzle.  dims/strides innermost
// first; strides are in bytes for dims 1..rank-1.  Returns false on failure.
bool encode_tmap_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box);
// The same for a one-byte element type (e4m3 operands).
bool encode_tmap_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

// ---------------------------------------------------------------------------------
// Launchers (each returns the launch's cudaError_t)
// ---------------------------------------------------------------------------------
struct AdaLNArgs {
  int batch, rows, hidden;
  const void* x;        // bf16, or fp32 when x_f32
  int x_f32;
  long long x_bstride;  // elements between batch rows of x
  int x_row0;
  bf16* y;
  long long y_bstride;
  int split;
  const bf16 *shift_lo, *scale_lo, *shift_hi, *scale_hi;
  long long mod_stride;  // elements between batch rows of the modulation vectors
  float eps;
  // Optional e4m3 output instead of y (bf16 x input only): y_q [batch, rows, hidden]
  // bytes (batch stride y_bstride) and one fp32 scale per row, y_scale [batch, rows].
  void* y_q;
  float* y_scale;
  // Status word for the kernel's bounded waits (may be null: a wait that gives up then only
  // ends the kernel early).
  DeviceStatus* status = nullptr;
};
bool adaln_supports(int hidden);  // hidden / 256 in {1..6, 8, 10, 12, 14, 16}
cudaError_t launch_adaln(const AdaLNArgs& a, cudaStream_t s);
// Per-row e4m3 quantisation of a bf16 weight [rows, cols]: q bytes, scale fp32 [rows].
cudaError_t launch_quantize_rows(const bf16* w, int rows, int cols, uint8_t* q, float* scale, cudaStream_t s);
// Per-row e4m3 quantisation of activations: rows of src (bf16; batch stride src_bstride,
// row stride ld, columns [col0, col0 + cols)) -> dst [batch, rows, cols] bytes and
// scale [batch * rows] = max|row| / 448.
bool quantize_act_supports(int cols);  // cols % 16 == 0 and cols <= 16384
cudaError_t launch_quantize_act(const bf16* src, long long src_bstride, int ld, int col0, int batch, int rows, int cols,
                                uint8_t* dst, float* scale, cudaStream_t s);

// y[b, n] = act(sum_k W[n, k] x[b, k]); x fp32 [batch, k]; W bf16 [n, k].
// act: 0 none, 1 SiLU.  Output fp32 (y_f32) or bf16 (y_bf16), exactly one non-null.
cudaError_t launch_gemv(const bf16* W, int n, int k, const float* x, int batch, int act, float* y_f32,
                        bf16* y_bf16, cudaStream_t s);
// SiLU(t_in * sinusoid(1000 sigma)) -> h [batch, H] fp32.
cudaError_t launch_timestep_in(const bf16* t_in, int H, int time_dim, const float* sigma, int batch, float* h,
                               cudaStream_t s);

// Denoising loop set-up: sigma[k*B + b] = sigmas[k], coef[k*B + b] = sigmas[k+1] - sigmas[k]
// for k < steps (sigmas: steps + 1 host values, steps <= 8).
cudaError_t launch_denoise_setup(const float* sigmas_host, int steps, int batch, float* sigma, float* coef,
                                 cudaStream_t s);

constexpr uint32_t kSelftestSite = 0x901;
cudaError_t launch_selftest_wait(DeviceStatus* status, unsigned long long limit_ns, cudaStream_t s);

cudaError_t launch_rope_table(const int32_t* ids, int n, const int* axes_dim, float theta, float* table,
                              cudaStream_t s);
cudaError_t launch_pack_mlp_in(const bf16* src, bf16* dst, int F, int cols, cudaStream_t s);

// ---------------------------------------------------------------------------------
// GEMM (tcgen05)
// ---------------------------------------------------------------------------------
enum EpiKind : int { kEpiStore = 0, kEpiResidual = 1, kEpiSwiGLU = 2, kEpiQKV = 3 };

struct GemmProblemHost {
  // A: [batch, a_rows_total, k] bf16 with row stride lda (elements), this problem uses
  // rows [a_row0, a_row0 + rows) of every batch slab.
  const bf16* a;
  int a_rows_total;
  long long lda;
  int a_row0;
  int rows;
  // W: [n, k] bf16 (row stride k).
  const bf16* w;
  int n, k;
  int epi;
  // STORE / RESIDUAL / SWIGLU destination: out + b*out_bstride + (out_row0 + r)*ld_out
  // + out_col0 + col.  RESIDUAL may write fp32 (out_f32, same addressing) instead of, or
  // as well as, bf16.
  bf16* out;
  float* out_f32;
  // RESIDUAL input x (same addressing as out): bf16 res or fp32 res_f32; may alias out.
  const bf16* res;
  const float* res_f32;
  long long out_bstride;
  int ld_out, out_row0, out_col0;
  // RESIDUAL gate vector (n entries at gate + b*gate_stride), or, when coef is set, one
  // fp32 coefficient per batch row (coef[b]) for every column.
  const bf16* gate;
  long long gate_stride;
  const float* coef;
  // e4m3 operands (fp8 != 0): A and W hold e4m3 bytes (lda in elements = bytes), the
  // product is dequantised in the epilogue by a_scale[b * a_rows_total + a_row] and
  // w_scale[col].  Every problem of one launch has the same fp8 setting.
  int fp8;
  const float* a_scale;
  const float* w_scale;
  // QKV: columns [0, n_qkv) are q | k | v (each `hidden` wide); columns >= n_qkv are a
  // packed SwiGLU pair written to `out` at out_col0 + (col - n_qkv) / 2.
  int n_qkv, hidden;
  bf16 *q, *kk, *v;         // [batch, heads, seq, 128]
  const bf16 *q_norm, *k_norm;
  const float* rope;        // [seq, 64, 2]
  int seq, tok0;            // token index of local row r is tok0 + r
};

cudaError_t launch_gemm(const GemmProblemHost* probs, int nprob, int batch, float eps, DeviceStatus* status,
                        int cls, cudaStream_t s);

// ---------------------------------------------------------------------------------
// Attention (tcgen05)
// ---------------------------------------------------------------------------------
cudaError_t launch_attention(int batch, int heads, int n, const bf16* q, const bf16* k, const bf16* v, bf16* out,
                             int ld_out, DeviceStatus* status, cudaStream_t s);

}  // namespace dit
