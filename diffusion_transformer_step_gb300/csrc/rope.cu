// RoPE table and MLP-in weight packing.
//
// RoPE ("tt_flux2_klein -- Python reference", "Things that are easy to get wrong"): four
// axes (t, h, w, l) of 32 dims each, theta 2000, rotations on adjacent pairs
// (repeat_interleave_real=True).  Axis a owns the head dims [off_a, off_a + dim_a); its
// pair j (dims off_a + 2j, off_a + 2j + 1) turns by pos_a * theta^(-2j / dim_a).  The
// table holds cos and sin of every pair angle, evaluated in fp64 and stored as fp32.
#include "runtime.h"

namespace dit {

namespace {

__global__ void rope_table_kernel(const int32_t* __restrict__ ids, int n, int4 axes, float theta,
                                  float* __restrict__ table) {
  const int pairs = (axes.x + axes.y + axes.z + axes.w) / 2;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)n * pairs) return;
  const int row = (int)(i / pairs);
  int p = (int)(i - (long long)row * pairs);
  const int dims[4] = {axes.x, axes.y, axes.z, axes.w};
  int a = 0;
  while (a < 3 && p >= dims[a] / 2) {
    p -= dims[a] / 2;
    ++a;
  }
  const double pos = (double)ids[(long long)row * 4 + a];
  const double omega = pow((double)theta, -2.0 * (double)p / (double)dims[a]);
  double s, c;
  sincos(pos * omega, &s, &c);
  table[2 * i] = (float)c;
  table[2 * i + 1] = (float)s;
}

// dst row r <- src row: block j = r / 256, within = r % 256; gate rows for within < 128.
__global__ void pack_mlp_in_kernel(const bf16* __restrict__ src, bf16* __restrict__ dst, int F, int cols) {
  const int r = blockIdx.x;
  const int j = r >> 8, w = r & 255;
  const int src_row = (w < 128) ? (j * 128 + w) : (F + j * 128 + (w - 128));
  const uint4* s = reinterpret_cast<const uint4*>(src + (long long)src_row * cols);
  uint4* d = reinterpret_cast<uint4*>(dst + (long long)r * cols);
  for (int c = threadIdx.x; c < cols / 8; c += blockDim.x) d[c] = s[c];
}

// Failure-detection self-test: one thread waits on an mbarrier that nothing arrives on,
// with a short limit; the bounded wait gives up, records the timeout and its site in the
// status word and the kernel returns normally.
__global__ void selftest_wait_kernel(DeviceStatus* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  const WaitCtx wc{status, &abort_flag, limit_ns};
  mbar_wait(&bar, 0, wc, kSelftestSite);
}

}  // namespace

cudaError_t launch_selftest_wait(DeviceStatus* status, unsigned long long limit_ns, cudaStream_t s) {
  LaunchScope scope(kClsRope, s);
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(const int32_t* ids, int n, const int* axes_dim, float theta, float* table,
                              cudaStream_t s) {
  const int pairs = (axes_dim[0] + axes_dim[1] + axes_dim[2] + axes_dim[3]) / 2;
  const long long total = (long long)n * pairs;
  if (total == 0) return cudaSuccess;
  const int block = 256;
  const unsigned grid = (unsigned)((total + block - 1) / block);
  LaunchScope scope(kClsRope, s);
  rope_table_kernel<<<grid, block, 0, s>>>(ids, n, make_int4(axes_dim[0], axes_dim[1], axes_dim[2], axes_dim[3]),
                                           theta, table);
  return cudaGetLastError();
}

cudaError_t launch_pack_mlp_in(const bf16* src, bf16* dst, int F, int cols, cudaStream_t s) {
  LaunchScope scope(kClsPack, s);
  pack_mlp_in_kernel<<<2 * F, 128, 0, s>>>(src, dst, F, cols);
  return cudaGetLastError();
}

}  // namespace dit
