// Adaptive LayerNorm with the per-step shift/scale: y = (1 + scale) LN(x) + shift.
// LayerNorm over the hidden dim without affine, biased variance, fp32 statistics
// (readings R3, R4).  Input rows are bf16, or fp32 for the dual-stream block's
// intermediate residual stream.  HBM-bound: each row is read once (2H or 4H bytes) and
// written once (2H bytes, or H bytes + a scale in e4m3); the modulation vectors stay in L1.
//
// Persistent streaming: one CTA per SM, one warp per row at a time.  Each warp owns a
// two-stage shared-memory ring: its lane 0 copies whole rows in with 1-D bulk copies
// (cp.async.bulk, completing on the stage's mbarrier), so the next row is in flight while
// the current one is reduced from shared memory (shifted sums with warp shuffles), then
// modulated and stored with 16-byte stores.
#include <cuda_fp8.h>

#include "runtime.h"

namespace dit {

namespace {

constexpr uint32_t kSiteAdaLN = 0x301;
constexpr int kMaxWarps = 16;
constexpr size_t kSmemBudget = 200 * 1024;

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Element k * 256 + 8 * lane + j (j < 8) of the staged row, as fp32 pairs.
template <bool F32IN>
__device__ __forceinline__ void load8(const uint8_t* buf, int k, int lane, float2 (&x)[4]) {
  if (F32IN) {
    const float4* xf = reinterpret_cast<const float4*>(buf) + 2 * (k * 32 + lane);
    const float4 f0 = xf[0], f1 = xf[1];
    x[0] = make_float2(f0.x, f0.y);
    x[1] = make_float2(f0.z, f0.w);
    x[2] = make_float2(f1.x, f1.y);
    x[3] = make_float2(f1.z, f1.w);
  } else {
    const uint4 u = reinterpret_cast<const uint4*>(buf)[k * 32 + lane];
    x[0] = unpack_bf16x2(u.x);
    x[1] = unpack_bf16x2(u.y);
    x[2] = unpack_bf16x2(u.z);
    x[3] = unpack_bf16x2(u.w);
  }
}

// kFp8Out: y is written as e4m3 with one fp32 scale per row (y ~ scale * q, scale =
// max|y| / 448, the largest finite e4m3), the A operand of an fp8 projection.
// The row stays in shared memory and is read once per pass: pass 1 the shifted sums
// (sum and sum of squares of x - x[0], exact enough in fp32 for any mean: the shift is a
// value of the row), pass 2 the modulated output (and, for e4m3, pass 2 the row maximum of
// y and pass 3 the codes).  Holding nothing of the row in registers lets 16 warps share an
// SM.  Packed fp32x2 arithmetic throughout.
template <int VPL, bool F32IN, bool kFp8Out>  // 8-element vectors per lane: hidden = VPL * 256
__global__ void __launch_bounds__(kMaxWarps * 32, 1) adaln_kernel(AdaLNArgs a) {
  constexpr int H = VPL * 256;
  constexpr uint32_t kRowBytes = (uint32_t)H * (F32IN ? 4u : 2u);
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ uint64_t bars[kMaxWarps][2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  uint8_t* buf0 = smem_raw + (size_t)(warp * 2) * kRowBytes;
  uint8_t* buf1 = buf0 + kRowBytes;
  uint64_t* bar = bars[warp];
  // Row indices in 32 bits (batch * rows <= 64 * 2^20 by the entry points' limits): the
  // per-row batch / row split is then a 32-bit division, not a 64-bit library routine.
  const int total = a.batch * a.rows;
  const int stride = (int)gridDim.x * nwarps;
  int r = (int)blockIdx.x * nwarps + warp;

  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
  }
  if (threadIdx.x == 0) abort_flag = 0;
  fence_mbar_init();
  __syncthreads();
  const WaitCtx wc{a.status, &abort_flag, kWaitLimitNs};
  grid_dependency_wait();  // x and y belong to earlier kernels of the stream
  allow_dependents();

  auto row_src = [&](int row) -> const uint8_t* {
    const int b = row / a.rows;
    const int rr = row - b * a.rows;
    return reinterpret_cast<const uint8_t*>(a.x) +
           (b * a.x_bstride + (long long)(a.x_row0 + rr) * H) * (F32IN ? 4 : 2);
  };
  int issued = 0;  // rows copied in by this warp (lane 0's count)
  if (lane == 0) {
    for (int st = 0; st < 2; ++st) {
      const int row = r + st * stride;
      if (row < total) {
        mbar_arrive_expect_tx(&bar[st], kRowBytes);
        bulk_copy_g2s(st ? buf1 : buf0, row_src(row), kRowBytes, &bar[st]);
        ++issued;
      }
    }
  }

  int consumed = 0;
  for (int i = 0; r < total; ++i, r += stride) {
    const int st = i & 1;
    bool ok = mbar_wait_sleep(&bar[st], (uint32_t)(i >> 1) & 1u, wc, kSiteAdaLN);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const uint8_t* buf = st ? buf1 : buf0;
    const int b = r / a.rows;
    const int rw = r - b * a.rows;

    // pass 1: shifted sums
    const float shift0 = F32IN ? reinterpret_cast<const float*>(buf)[0]
                               : __bfloat162float(reinterpret_cast<const bf16*>(buf)[0]);
    const float2 nk = make_float2(-shift0, -shift0);
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int k = 0; k < VPL; ++k) {
      float2 x[4];
      load8<F32IN>(buf, k, lane, x);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 d = __fadd2_rn(x[j], nk);
        s1 = __fadd2_rn(s1, d);
        s2 = __ffma2_rn(d, d, s2);
      }
    }
    float sum = s1.x + s1.y, sq = s2.x + s2.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum += __shfl_xor_sync(0xffffffffu, sum, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
    }
    const float dm = sum * (1.0f / H);  // mean - shift0
    const float var = fmaxf(sq * (1.0f / H) - dm * dm, 0.f);
    const float rstd = rsqrtf(var + a.eps);
    const float mean = shift0 + dm;
    // n = x * rstd - mean * rstd
    const float2 rs2 = make_float2(rstd, rstd), mb2 = make_float2(-mean * rstd, -mean * rstd);
    const float2 one = make_float2(1.f, 1.f);

    const bool lo = rw < a.split;
    const uint4* shv = reinterpret_cast<const uint4*>((lo ? a.shift_lo : a.shift_hi) + b * a.mod_stride);
    const uint4* scv = reinterpret_cast<const uint4*>((lo ? a.scale_lo : a.scale_hi) + b * a.mod_stride);
    // y for the 8 elements of vector k of this lane
    auto modulated = [&](int k, float2 (&y)[4]) {
      float2 x[4];
      load8<F32IN>(buf, k, lane, x);
      const uint4 sh = __ldg(shv + k * 32 + lane);
      const uint4 sc = __ldg(scv + k * 32 + lane);
      const uint32_t shw[4] = {sh.x, sh.y, sh.z, sh.w};
      const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 n = __ffma2_rn(x[j], rs2, mb2);
        y[j] = __ffma2_rn(__fadd2_rn(unpack_bf16x2(scw[j]), one), n, unpack_bf16x2(shw[j]));
      }
    };

    if (!kFp8Out) {
      uint4* yv = reinterpret_cast<uint4*>(a.y + b * a.y_bstride + (long long)rw * H);
#pragma unroll 4
      for (int k = 0; k < VPL; ++k) {
        float2 y[4];
        modulated(k, y);
        yv[k * 32 + lane] = make_uint4(pack_bf16x2(y[0].x, y[0].y), pack_bf16x2(y[1].x, y[1].y),
                                       pack_bf16x2(y[2].x, y[2].y), pack_bf16x2(y[3].x, y[3].y));
      }
    } else {
      float amax = 0.f;
#pragma unroll 4
      for (int k = 0; k < VPL; ++k) {
        float2 y[4];
        modulated(k, y);
#pragma unroll
        for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fmaxf(fabsf(y[j].x), fabsf(y[j].y)));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float scale = amax > 0.f ? amax / 448.0f : 1.0f;
      const float inv = 1.0f / scale;
      uint2* qv = reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(a.y_q) + b * a.y_bstride + (long long)rw * H);
#pragma unroll 4
      for (int k = 0; k < VPL; ++k) {
        float2 y[4];
        modulated(k, y);
        uint32_t w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const __nv_fp8x2_storage_t q0 =
              __nv_cvt_float2_to_fp8x2(make_float2(y[2 * h].x * inv, y[2 * h].y * inv), __NV_SATFINITE, __NV_E4M3);
          const __nv_fp8x2_storage_t q1 = __nv_cvt_float2_to_fp8x2(
              make_float2(y[2 * h + 1].x * inv, y[2 * h + 1].y * inv), __NV_SATFINITE, __NV_E4M3);
          w[h] = (uint32_t)q0 | ((uint32_t)q1 << 16);
        }
        qv[k * 32 + lane] = make_uint2(w[0], w[1]);
      }
      if (lane == 0) a.y_scale[(long long)b * a.rows + rw] = scale;
    }
    ++consumed;
    // every lane has finished reading the staged row: the stage may be refilled (the
    // generic-proxy reads are ordered before the bulk copy's async-proxy writes)
    __syncwarp();
    if (lane == 0) {
      fence_proxy_async_smem();
      const int nrow = r + 2 * stride;
      if (nrow < total) {
        mbar_arrive_expect_tx(&bar[st], kRowBytes);
        bulk_copy_g2s(st ? buf1 : buf0, row_src(nrow), kRowBytes, &bar[st]);
        ++issued;
      }
    }
  }
  // After an early exit, let this warp's copies still in flight land (bounded) before the
  // block's shared memory is released.
  if (lane == 0) {
    const uint64_t t0 = global_timer_ns();
    for (int k = consumed; k < issued; ++k)
      while (!mbar_try(&bar[k & 1], (uint32_t)(k >> 1) & 1u) && global_timer_ns() - t0 < 100000000ull) {
      }
  }
}

// Per-row e4m3 quantisation of a weight: scale[r] = max|w[r, :]| / 448, q = w / scale.
__global__ void quantize_rows_kernel(const bf16* __restrict__ w, int cols, uint8_t* __restrict__ q,
                                     float* __restrict__ scale) {
  const int r = blockIdx.x;
  const bf16* wr = w + (long long)r * cols;
  float amax = 0.f;
  for (int c = threadIdx.x; c < cols; c += blockDim.x) amax = fmaxf(amax, fabsf(__bfloat162float(wr[c])));
  __shared__ float red[32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    amax = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (threadIdx.x == 0) red[0] = amax;
  }
  __syncthreads();
  const float s = red[0] > 0.f ? red[0] / 448.0f : 1.0f;
  const float inv = 1.0f / s;
  for (int c = threadIdx.x; c < cols; c += blockDim.x)
    q[(long long)r * cols + c] = (uint8_t)__nv_cvt_float_to_fp8(__bfloat162float(wr[c]) * inv, __NV_SATFINITE, __NV_E4M3);
  if (threadIdx.x == 0) scale[r] = s;
}

// Per-row e4m3 quantisation of activations (the A operand of an e4m3 out-projection):
// row r of src (bf16, batch stride src_bstride, row stride ld, columns [col0, col0 + cols))
// -> dst[r, :] (cols bytes, rows contiguous) and scale[r] = max|row| / 448.  One CTA per row,
// the row held in registers (up to kMaxVec 8-element vectors per thread): one read, one write.
constexpr int kQuantThreads = 256, kQuantMaxVec = 8;

__global__ void __launch_bounds__(kQuantThreads) quantize_act_kernel(const bf16* __restrict__ src,
                                                                     long long src_bstride, int ld, int col0, int rows,
                                                                     int cols, uint8_t* __restrict__ dst,
                                                                     float* __restrict__ scale) {
  grid_dependency_wait();  // src and dst belong to earlier kernels of the stream
  allow_dependents();
  const long long row = blockIdx.x;  // batch * rows
  const int b = (int)(row / rows);
  const int r = (int)(row - (long long)b * rows);
  const uint4* s4 = reinterpret_cast<const uint4*>(src + b * src_bstride + (long long)r * ld + col0);
  const int nvec = cols >> 3;
  uint4 v[kQuantMaxVec];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kQuantMaxVec; ++i) {
    const int idx = threadIdx.x + i * kQuantThreads;
    if (idx < nvec) {
      v[i] = __ldg(s4 + idx);
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = unpack_bf16x2(w[j]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
  }
  __shared__ float red[kQuantThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < kQuantThreads / 32; ++i) amax = fmaxf(amax, red[i]);
  const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
  const float inv = 1.0f / sc;
  uint2* d2 = reinterpret_cast<uint2*>(dst + row * cols);
#pragma unroll
  for (int i = 0; i < kQuantMaxVec; ++i) {
    const int idx = threadIdx.x + i * kQuantThreads;
    if (idx < nvec) {
      const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
      uint32_t q[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float2 f0 = unpack_bf16x2(w[2 * h]), f1 = unpack_bf16x2(w[2 * h + 1]);
        const __nv_fp8x2_storage_t q0 =
            __nv_cvt_float2_to_fp8x2(make_float2(f0.x * inv, f0.y * inv), __NV_SATFINITE, __NV_E4M3);
        const __nv_fp8x2_storage_t q1 =
            __nv_cvt_float2_to_fp8x2(make_float2(f1.x * inv, f1.y * inv), __NV_SATFINITE, __NV_E4M3);
        q[h] = (uint32_t)q0 | ((uint32_t)q1 << 16);
      }
      d2[idx] = make_uint2(q[0], q[1]);
    }
  }
  if (threadIdx.x == 0) scale[row] = sc;
}

template <int VPL, bool F32IN, bool kFp8Out>
cudaError_t launch_kind(const AdaLNArgs& a, cudaStream_t s) {
  const size_t row_bytes = (size_t)VPL * 256 * (F32IN ? 4 : 2);
  int warps = (int)(kSmemBudget / (2 * row_bytes));
  if (warps > kMaxWarps) warps = kMaxWarps;
  const size_t smem = (size_t)warps * 2 * row_bytes;
  // One CTA per SM with as many warps as two staged rows each allow in the shared-memory
  // budget (16 for bf16 rows of 3072, 8 for fp32 ones): up to 32 rows in flight per SM.
  const long long total = (long long)a.batch * a.rows;
  long long grid = (total + warps - 1) / warps;
  const long long cap = (long long)sm_count();
  if (grid > cap) grid = cap;
  auto k = adaln_kernel<VPL, F32IN, kFp8Out>;
  // The static shared memory (row barriers and the abort flag, under 1 KB) counts against
  // the same 48 KB default as the dynamic part: hidden 768 asks for exactly 48 KB dynamic.
  if (smem + 1024 > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  LaunchScope scope(kClsAdaLN, s);
  return launch_k(k, dim3((unsigned)grid), dim3(warps * 32), smem, s, a);
}

template <int VPL>
cudaError_t launch_vpl(const AdaLNArgs& a, cudaStream_t s) {
  if (a.y_q) return a.x_f32 ? launch_kind<VPL, true, true>(a, s) : launch_kind<VPL, false, true>(a, s);
  if (a.x_f32) return launch_kind<VPL, true, false>(a, s);
  return launch_kind<VPL, false, false>(a, s);
}

}  // namespace

bool adaln_supports(int hidden) {
  if (hidden <= 0 || hidden % 256 != 0) return false;
  switch (hidden / 256) {
    case 1: case 2: case 3: case 4: case 5: case 6: case 8: case 10: case 12: case 14: case 16: return true;
    default: return false;
  }
}

cudaError_t launch_adaln(const AdaLNArgs& a, cudaStream_t s) {
  if ((long long)a.batch * a.rows == 0) return cudaSuccess;
  if ((long long)a.batch * a.rows > (1ll << 26)) return cudaErrorInvalidValue;  // the kernel's 32-bit row index
  switch (a.hidden / 256) {
    case 1: return launch_vpl<1>(a, s);
    case 2: return launch_vpl<2>(a, s);
    case 3: return launch_vpl<3>(a, s);
    case 4: return launch_vpl<4>(a, s);
    case 5: return launch_vpl<5>(a, s);
    case 6: return launch_vpl<6>(a, s);
    case 8: return launch_vpl<8>(a, s);
    case 10: return launch_vpl<10>(a, s);
    case 12: return launch_vpl<12>(a, s);
    case 14: return launch_vpl<14>(a, s);
    case 16: return launch_vpl<16>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dit

namespace dit {
cudaError_t launch_quantize_rows(const bf16* w, int rows, int cols, uint8_t* q, float* scale, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  LaunchScope scope(kClsPack, s);
  quantize_rows_kernel<<<rows, 256, 0, s>>>(w, cols, q, scale);
  return cudaGetLastError();
}
}  // namespace dit

namespace dit {
bool quantize_act_supports(int cols) { return cols > 0 && cols % 16 == 0 && cols / 8 <= kQuantThreads * kQuantMaxVec; }

cudaError_t launch_quantize_act(const bf16* src, long long src_bstride, int ld, int col0, int batch, int rows, int cols,
                                uint8_t* dst, float* scale, cudaStream_t s) {
  if ((long long)batch * rows == 0) return cudaSuccess;
  if (!quantize_act_supports(cols)) return cudaErrorInvalidValue;
  LaunchScope scope(kClsQuantAct, s);
  return launch_k(quantize_act_kernel, dim3((unsigned)((long long)batch * rows)), dim3(kQuantThreads), 0, s, src,
                  src_bstride, ld, col0, rows, cols, dst, scale);
}
}  // namespace dit
