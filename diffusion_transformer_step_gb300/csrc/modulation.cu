// The global per-step modulation ("flux2-klein-p100a" model card, Caveats: modulation
// is global per step, not per block): a timestep MLP followed by one projection to all
// 17 shift / scale / gate vectors.  With batch <= 8 these are matrix-vector products that
// read each weight once: HBM-bound GEMVs on the CUDA cores, one warp per output row,
// 128-bit weight loads, the input vectors held in shared memory.
#include "runtime.h"

namespace dit {

namespace {

constexpr int kWarps = 8;
constexpr int kMaxBatchPerLaunch = 8;

template <int NB>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(const bf16* __restrict__ W, int n, int k,
                                                            const float* __restrict__ x, int act,
                                                            float* __restrict__ y_f32, bf16* __restrict__ y_bf16,
                                                            int y_stride) {
  extern __shared__ float xs[];  // [NB][k]
  grid_dependency_wait();
  allow_dependents();
  for (int i = threadIdx.x; i < NB * k; i += blockDim.x) xs[i] = x[i];
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = k >> 3;
  for (int row = blockIdx.x * kWarps + warp; row < n; row += gridDim.x * kWarps) {
    const uint4* wr = reinterpret_cast<const uint4*>(W + (long long)row * k);
    float acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = 0.f;
#pragma unroll 4
    for (int v = lane; v < nvec; v += 32) {
      const uint4 u = __ldg(wr + v);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
      float wf[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = unpack_bf16x2(w4[j]);
        wf[2 * j] = f.x;
        wf[2 * j + 1] = f.y;
      }
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float4 x0 = *reinterpret_cast<const float4*>(xs + b * k + v * 8);
        const float4 x1 = *reinterpret_cast<const float4*>(xs + b * k + v * 8 + 4);
        acc[b] += wf[0] * x0.x + wf[1] * x0.y + wf[2] * x0.z + wf[3] * x0.w + wf[4] * x1.x + wf[5] * x1.y +
                  wf[6] * x1.z + wf[7] * x1.w;
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float s = acc[b];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) {
        if (act == 1) s = s / (1.0f + expf(-s));
        if (y_f32) y_f32[(long long)b * y_stride + row] = s;
        else y_bf16[(long long)b * y_stride + row] = __float2bfloat16_rn(s);
      }
    }
  }
}

// h[b, n] = SiLU(sum_k t_in[n, k] s_b[k]); s_b = [cos(1000 sigma_b f_k) | sin(...)],
// f_k = 10000^(-k / (time_dim/2)).  The sinusoid is evaluated in fp64.
__global__ void __launch_bounds__(kWarps * 32) timestep_in_kernel(const bf16* __restrict__ t_in, int H,
                                                                   int time_dim, const float* __restrict__ sigma,
                                                                   int batch, float* __restrict__ h) {
  extern __shared__ float sv[];  // [batch][time_dim]
  grid_dependency_wait();
  allow_dependents();
  const int half = time_dim / 2;
  for (int i = threadIdx.x; i < batch * half; i += blockDim.x) {
    const int b = i / half, kk = i - b * half;
    const double tau = 1000.0 * (double)sigma[b];
    const double f = exp(-log(10000.0) * (double)kk / (double)half);
    double s, c;
    sincos(tau * f, &s, &c);
    sv[b * time_dim + kk] = (float)c;
    sv[b * time_dim + half + kk] = (float)s;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int row = blockIdx.x * kWarps + warp; row < H; row += gridDim.x * kWarps) {
    const bf16* wr = t_in + (long long)row * time_dim;
    for (int b = 0; b < batch; ++b) {
      float acc = 0.f;
      for (int kk = lane; kk < time_dim; kk += 32) acc += __bfloat162float(wr[kk]) * sv[b * time_dim + kk];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (lane == 0) h[(long long)b * H + row] = acc / (1.0f + expf(-acc));
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

template <int NB>
cudaError_t gemv_nb(const bf16* W, int n, int k, const float* x, int act, float* y_f32, bf16* y_bf16, int y_stride,
                    cudaStream_t s) {
  const size_t smem = (size_t)NB * k * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int grid = (n + kWarps - 1) / kWarps;
  const int cap = sm_count() * 8;
  if (grid > cap) grid = cap;
  LaunchScope scope(kClsModulation, s);
  return launch_k(gemv_kernel<NB>, dim3(grid), dim3(kWarps * 32), smem, s, W, n, k, x, act, y_f32, y_bf16, y_stride);
}

}  // namespace

cudaError_t launch_gemv(const bf16* W, int n, int k, const float* x, int batch, int act, float* y_f32,
                        bf16* y_bf16, cudaStream_t s) {
  for (int b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
    const int nb = batch - b0 < kMaxBatchPerLaunch ? batch - b0 : kMaxBatchPerLaunch;
    const float* xb = x + (long long)b0 * k;
    float* yf = y_f32 ? y_f32 + (long long)b0 * n : nullptr;
    bf16* yb = y_bf16 ? y_bf16 + (long long)b0 * n : nullptr;
    cudaError_t e;
    switch (nb) {
      case 1: e = gemv_nb<1>(W, n, k, xb, act, yf, yb, n, s); break;
      case 2: e = gemv_nb<2>(W, n, k, xb, act, yf, yb, n, s); break;
      case 3: e = gemv_nb<3>(W, n, k, xb, act, yf, yb, n, s); break;
      case 4: e = gemv_nb<4>(W, n, k, xb, act, yf, yb, n, s); break;
      case 5: e = gemv_nb<5>(W, n, k, xb, act, yf, yb, n, s); break;
      case 6: e = gemv_nb<6>(W, n, k, xb, act, yf, yb, n, s); break;
      case 7: e = gemv_nb<7>(W, n, k, xb, act, yf, yb, n, s); break;
      default: e = gemv_nb<8>(W, n, k, xb, act, yf, yb, n, s); break;
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
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
  const size_t smem = (size_t)batch * time_dim * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(timestep_in_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int grid = (H + kWarps - 1) / kWarps;
  const int cap = sm_count() * 4;
  if (grid > cap) grid = cap;
  LaunchScope scope(kClsModulation, s);
  return launch_k(timestep_in_kernel, dim3(grid), dim3(kWarps * 32), smem, s, t_in, H, time_dim, sigma, batch, h);
}

}  // namespace dit
