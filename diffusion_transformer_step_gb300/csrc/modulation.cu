// The global per-step modulation ("flux2-klein-p100a" model card, Caveats: modulation
// is global per step, not per block): a timestep MLP followed by one projection to all
// 17 shift / scale / gate vectors.  With batch <= 8 these are matrix-vector products that
// read each weight once: HBM-bound GEMVs on the CUDA cores.
//
// One GEMV kernel serves all three products.  The grid is persistent: as many CTAs as fit
// on the GPU at once (one wave), each warp walking pairs of weight rows.  A lane owns the
// same 8-element slices of every row (slice c covers columns [256c + 8 lane, +8)), so
// its input values come from shared memory once per slice and feed both rows of the
// pair.  Each lane keeps 2 x kChunks 16-byte weight loads in flight (streamed past L1),
// accumulates with packed fp32x2 FMAs and the pair's sums meet in a warp-shuffle
// reduction.  The first product (the timestep MLP's input layer) computes its input, the
// sinusoid of 1000 sigma, in each CTA's prologue: the angle is formed and reduced modulo
// 2 pi in fp64 (tau * f_k / pi - 2 round(tau * f_k / 2 pi)), then sin and cos of pi times
// the reduced value are taken in fp32.
#include <math.h>

#include <atomic>

#include "runtime.h"

namespace dit {

namespace {

constexpr int kWarps = 8;
constexpr int kChunks = 4;             // 16-byte loads in flight per row and lane
constexpr int kMaxBatchPerLaunch = 8;
constexpr int kMaxTimeHalf = 128;      // sinusoid width / 2 (the modulation uses 256)

// f_k / pi = 10000^(-k / half) / pi for k < half, evaluated on the host in fp64.
struct SinusoidFreqs {
  double g[kMaxTimeHalf];
  int half;
};

__device__ __forceinline__ uint4 ld_stream16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Both rows' 8 weights of one slice against the NB input vectors at xv (stride k).
template <int NB>
__device__ __forceinline__ void slice_fma(const uint4& u0, const uint4& u1, const float* xv, int k, float2 (&a0)[NB],
                                          float2 (&a1)[NB]) {
  const float2 w0[4] = {unpack_bf16x2(u0.x), unpack_bf16x2(u0.y), unpack_bf16x2(u0.z), unpack_bf16x2(u0.w)};
  const float2 w1[4] = {unpack_bf16x2(u1.x), unpack_bf16x2(u1.y), unpack_bf16x2(u1.z), unpack_bf16x2(u1.w)};
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const float4 xa = *reinterpret_cast<const float4*>(xv + b * k);
    const float4 xb = *reinterpret_cast<const float4*>(xv + b * k + 4);
    const float2 x2[4] = {make_float2(xa.x, xa.y), make_float2(xa.z, xa.w), make_float2(xb.x, xb.y),
                          make_float2(xb.z, xb.w)};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      a0[b] = __ffma2_rn(w0[j], x2[j], a0[b]);
      a1[b] = __ffma2_rn(w1[j], x2[j], a1[b]);
    }
  }
}

// y[b, r] = act(sum_c W[r, c] x[b, c]) for rows r < n; k % 256 == 0.  x is either the fp32
// input [NB, k] (kSinusoid false) or, for the timestep layer (k = 2 * half), the
// sinusoid [cos(tau_b f_c) | sin(tau_b f_c)] of tau_b = 1000 sigma[b].
template <int NB, bool kSinusoid>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(const bf16* __restrict__ W, int n, int k,
                                                            const float* __restrict__ x, const SinusoidFreqs fr,
                                                            int act, float* __restrict__ y_f32,
                                                            bf16* __restrict__ y_bf16, int y_stride) {
  extern __shared__ __align__(16) float xs[];  // [NB][k]
  grid_dependency_wait();  // x (or sigma) comes from an earlier kernel; y is read by later ones
  allow_dependents();
  if (kSinusoid) {
    for (int i = threadIdx.x; i < NB * fr.half; i += blockDim.x) {
      const int b = i / fr.half, c = i - b * fr.half;
      const double t = 1000.0 * (double)x[b] * fr.g[c];  // angle / pi
      const double r = t - 2.0 * rint(0.5 * t);          // in [-1, 1]: angle mod 2 pi, over pi
      float sv, cv;
      sincospif((float)r, &sv, &cv);
      xs[b * k + c] = cv;
      xs[b * k + fr.half + c] = sv;
    }
  } else {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    for (int i = threadIdx.x; i < NB * k / 4; i += blockDim.x) reinterpret_cast<float4*>(xs)[i] = x4[i];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nslice = k >> 8;
  const int npairs = (n + 1) >> 1;
  for (int pr = blockIdx.x * kWarps + warp; pr < npairs; pr += gridDim.x * kWarps) {
    const int r0 = 2 * pr, r1 = r0 + 1 < n ? r0 + 1 : r0;  // a lone last row is read twice, stored once
    const uint4* w0 = reinterpret_cast<const uint4*>(W + (long long)r0 * k) + lane;
    const uint4* w1 = reinterpret_cast<const uint4*>(W + (long long)r1 * k) + lane;
    float2 a0[NB], a1[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) a0[b] = a1[b] = make_float2(0.f, 0.f);
    for (int c0 = 0; c0 < nslice; c0 += kChunks) {
      uint4 u0[kChunks], u1[kChunks];
#pragma unroll
      for (int g = 0; g < kChunks; ++g)
        if (c0 + g < nslice) {
          u0[g] = ld_stream16(w0 + (c0 + g) * 32);
          u1[g] = ld_stream16(w1 + (c0 + g) * 32);
        }
#pragma unroll
      for (int g = 0; g < kChunks; ++g)
        if (c0 + g < nslice) slice_fma<NB>(u0[g], u1[g], xs + (c0 + g) * 256 + lane * 8, k, a0, a1);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float s0 = a0[b].x + a0[b].y, s1 = a1[b].x + a1[b].y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      }
      if (lane < 2 && (lane == 0 || r1 != r0)) {
        float s = lane ? s1 : s0;
        const int row = lane ? r1 : r0;
        if (act == 1) s = s / (1.0f + expf(-s));
        if (y_f32) y_f32[(long long)b * y_stride + row] = s;
        else y_bf16[(long long)b * y_stride + row] = __float2bfloat16_rn(s);
      }
    }
  }
}

struct SigmaList {
  float v[9];
};

__global__ void denoise_setup_kernel(SigmaList sl, int steps, int batch, float* __restrict__ sigma,
                                     float* __restrict__ coef) {
  grid_dependency_wait();
  allow_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= steps * batch) return;
  const int k = i / batch;
  sigma[i] = sl.v[k];
  coef[i] = sl.v[k + 1] - sl.v[k];
}

// CTAs of gemv_kernel<NB, S> resident per SM with `smem` bytes of shared memory each,
// cached per device and instantiation together with the size it was computed for.
template <int NB, bool S>
int resident_ctas(size_t smem) {
  static std::atomic<unsigned long long> cached[16];  // (smem << 32) | count
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 16) {
    const unsigned long long c = cached[dev].load(std::memory_order_relaxed);
    if (c != 0 && (c >> 32) == (unsigned long long)smem) return (int)(c & 0xffffffffu);
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_kernel<NB, S>, kWarps * 32, smem) != cudaSuccess ||
      n < 1) {
    cudaGetLastError();
    n = 1;
  }
  if (dev >= 0 && dev < 16) cached[dev].store(((unsigned long long)smem << 32) | (unsigned)n, std::memory_order_relaxed);
  return n;
}

template <int NB, bool S>
cudaError_t gemv_nb(const bf16* W, int n, int k, const float* x, const SinusoidFreqs& fr, int act, float* y_f32,
                    bf16* y_bf16, int y_stride, cudaStream_t s) {
  const size_t smem = (size_t)NB * k * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NB, S>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // one wave of persistent CTAs, no more than the row pairs need
  const int need = ((n + 1) / 2 + kWarps - 1) / kWarps;
  const int cap = sm_count() * resident_ctas<NB, S>(smem);
  const int grid = need < cap ? need : cap;
  LaunchScope scope(kClsModulation, s);
  return launch_k(gemv_kernel<NB, S>, dim3(grid), dim3(kWarps * 32), smem, s, W, n, k, x, fr, act, y_f32, y_bf16,
                  y_stride);
}

template <bool S>
cudaError_t gemv_batched(const bf16* W, int n, int k, const float* x, int x_stride, const SinusoidFreqs& fr,
                         int batch, int act, float* y_f32, bf16* y_bf16, cudaStream_t s) {
  for (int b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
    const int nb = batch - b0 < kMaxBatchPerLaunch ? batch - b0 : kMaxBatchPerLaunch;
    const float* xb = x + (long long)b0 * x_stride;
    float* yf = y_f32 ? y_f32 + (long long)b0 * n : nullptr;
    bf16* yb = y_bf16 ? y_bf16 + (long long)b0 * n : nullptr;
    cudaError_t e;
    switch (nb) {
      case 1: e = gemv_nb<1, S>(W, n, k, xb, fr, act, yf, yb, n, s); break;
      case 2: e = gemv_nb<2, S>(W, n, k, xb, fr, act, yf, yb, n, s); break;
      case 3: e = gemv_nb<3, S>(W, n, k, xb, fr, act, yf, yb, n, s); break;
      case 4: e = gemv_nb<4, S>(W, n, k, xb, fr, act, yf, yb, n, s); break;
      case 5: e = gemv_nb<5, S>(W, n, k, xb, fr, act, yf, yb, n, s); break;
      case 6: e = gemv_nb<6, S>(W, n, k, xb, fr, act, yf, yb, n, s); break;
      case 7: e = gemv_nb<7, S>(W, n, k, xb, fr, act, yf, yb, n, s); break;
      default: e = gemv_nb<8, S>(W, n, k, xb, fr, act, yf, yb, n, s); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemv(const bf16* W, int n, int k, const float* x, int batch, int act, float* y_f32,
                        bf16* y_bf16, cudaStream_t s) {
  if (k <= 0 || k % 256 != 0) return cudaErrorInvalidValue;
  SinusoidFreqs unused;
  unused.half = 0;
  return gemv_batched<false>(W, n, k, x, k, unused, batch, act, y_f32, y_bf16, s);
}

cudaError_t launch_denoise_setup(const float* sigmas_host, int steps, int batch, float* sigma, float* coef,
                                 cudaStream_t s) {
  if (steps < 1 || steps > 8) return cudaErrorInvalidValue;
  SigmaList sl;
  for (int k = 0; k <= steps; ++k) sl.v[k] = sigmas_host[k];
  const int n = steps * batch;
  LaunchScope scope(kClsModulation, s);
  return launch_k(denoise_setup_kernel, dim3((n + 127) / 128), dim3(128), 0, s, sl, steps, batch, sigma, coef);
}

cudaError_t launch_timestep_in(const bf16* t_in, int H, int time_dim, const float* sigma, int batch, float* h,
                               cudaStream_t s) {
  if (time_dim % 256 != 0 || time_dim / 2 > kMaxTimeHalf) return cudaErrorInvalidValue;
  SinusoidFreqs fr;
  fr.half = time_dim / 2;
  for (int c = 0; c < fr.half; ++c) fr.g[c] = exp(-log(10000.0) * (double)c / (double)fr.half) / M_PI;
  // sigma [batch] is read one value per batch row: x_stride 1
  return gemv_batched<true>(t_in, H, time_dim, sigma, 1, fr, batch, 1, h, nullptr, s);
}

}  // namespace dit
