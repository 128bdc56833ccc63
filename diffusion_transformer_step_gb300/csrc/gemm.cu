// Persistent tcgen05 GEMM with fused epilogues: out = A W^T, A [rows, k] and W [n, k]
// both K-major bf16, fp32 accumulation in Tensor Memory.
//
// CTA pairs (clusters of 2, tcgen05 cta_group::2), one CTA per SM, 320 threads each.  A
// pair computes a 256 x 256 tile: CTA r loads rows [128r, 128r + 128) of the A tile and
// rows [128r, 128r + 128) of the W tile, so each CTA streams 32 KB per 64-deep k-block
// (a 1-CTA 128 x 256 tile needs 48 KB for half the work) and 7 stages fit in shared memory
// (230 656 of the 232 448 bytes a CTA may have).  A timestamp trace showed the MMA issuer
// waiting for TMA data 16-19 % of each main loop with 6 stages; the seventh cut that by a
// tenth and the main loops by 2-4 %.
//   warp 0      TMA producer in both CTAs: 128-byte-swizzled tiles into a 7-stage ring;
//               both CTAs' loads complete on the leader CTA's full barrier, and the CTA
//               owning the first M tile of a weight column prefetches that column's W tiles
//               8 k-blocks ahead into L2 (one prefetcher per column, not every reader);
//   warp 1      allocates 512 TMEM columns in both CTAs (two 128 x 256 fp32 accumulators
//               per CTA) and, in the leader only, issues tcgen05.mma.cta_group::2 (M=256,
//               N=256, K=16) from one thread; commits are multicast to both CTAs' empty
//               and accumulator-full barriers;
//   warps 2-9   epilogue in both CTAs: two warps per TMEM lane quarter, each taking one
//               128-column half of the accumulator (one QKV head, one half of the SwiGLU
//               outputs, four 32-column chunks of a residual or plain store), one thread per
//               accumulator row of its own CTA, tcgen05.ld 32 columns at a time, fused math,
//               16-byte global stores; the accumulator is handed back on the leader's
//               barrier (16 arrivals).  Two warps per row keep a tile's epilogue shorter
//               than the next tile's main loop even for K = 3072 with an fp32 residual
//               output, where one warp per row (its loads of the residual serialised chunk
//               by chunk) took 18 us against a 14.5 us main loop and held the MMAs back.
// The two accumulators let tile i's epilogue overlap tile i+1's main loop.  Because the
// MMA-issuing warp competes for issue slots with the epilogue warp of its SM sub-partition
// (on sm_103a dense scalar FP32 FMA there slows tcgen05.mma issue several-fold, packed
// fp32x2 arithmetic does not), the epilogue maths runs on packed fp32x2 FMA / multiply / add
// with MUFU exponentials and reciprocals, the issuer advances precomputed descriptors with
// one add per MMA, and waiting warps sleep on their barriers.  Up to two
// problems (the text and image streams of a dual-stream block) share one launch; tiles
// are ordered with M fastest so that concurrent pairs share the same weight slab in L2.
//
// Epilogues (the fused block maths):
//   STORE     bf16(acc)
//   RESIDUAL  out <- x + gate * acc  (gated residual, reading R4); x and out bf16 or
//             fp32 (or both outputs), possibly the same buffer; the gate is a bf16 vector
//             per batch row, or one fp32 scalar per batch row (the Euler update
//             x + (sigma_next - sigma) v of the denoising loop)
//   SWIGLU    silu(acc[gate cols]) * acc[up cols]          (reading R9; packed W rows)
//   QKV       columns [0, 3H): per-head RMSNorm (fp32, eps) * w, RoPE on adjacent pairs
//             from the fp32 table, written head-major [B, heads, seq, 128]; columns
//             >= 3H: SWIGLU into the concat buffer (single-stream fused projection).
#include <atomic>

#include "runtime.h"

namespace dit {

namespace {

constexpr int BM = 128, BN = 256, BK = 64;   // per CTA: 128 rows of A; the pair's tile is 256 x 256
constexpr int PAIR_M = 2 * BM;
constexpr int kStages = 7;
constexpr int kThreads = 320;
constexpr uint32_t kATileBytes = BM * BK * 2;        // 16 KB (this CTA's half of A)
constexpr uint32_t kBTileBytes = (BN / 2) * BK * 2;  // 16 KB (this CTA's half of B)
constexpr uint32_t kStageBytes = kATileBytes + kBTileBytes;
constexpr uint32_t kTmemCols = 2 * BN;
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + 256;

struct DevProblem {
  int rows, a_row0, n, k, m_tiles, n_tiles, tile_begin, epi;
  bf16* out;
  float* out_f32;
  const bf16* res;
  const float* res_f32;
  long long out_bstride;
  int ld_out, out_row0, out_col0;
  const bf16* gate;
  long long gate_stride;
  const float* coef;
  const float* a_scale;     // fp8 operands: per-row activation scales (row b*a_rows_total + a_row)
  const float* w_scale;     // fp8 operands: per-output-column weight scales
  int a_rows_total;
  int n_qkv, hidden;
  bf16 *q, *kk, *v;
  const bf16 *q_norm, *k_norm;
  const float* rope;
  int seq, tok0;
};

struct alignas(64) GemmParams {
  CUtensorMap a_map[2];
  CUtensorMap b_map[2];
  DevProblem prob[2];
  int nprob, batch, total_tiles;
  float eps;
  DeviceStatus* status;
};

struct TileInfo {
  int p, b, m_tile, n_tile;
};

__device__ __forceinline__ TileInfo decode_tile(const GemmParams& P, int t) {
  TileInfo ti;
  ti.p = (P.nprob > 1 && t >= P.prob[1].tile_begin) ? 1 : 0;
  const DevProblem& pr = P.prob[ti.p];
  const int local = t - pr.tile_begin;
  const int per_b = pr.m_tiles * pr.n_tiles;
  ti.b = local / per_b;
  const int r = local - ti.b * per_b;
  ti.n_tile = r / pr.m_tiles;
  ti.m_tile = r - ti.n_tile * pr.m_tiles;
  return ti;
}

// Wait sites, reported through DeviceStatus::where.
enum : uint32_t { kSiteEmpty = 0x101, kSiteFull = 0x102, kSiteAccEmpty = 0x103, kSiteAccFull = 0x104 };

__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}
__device__ __forceinline__ void tma3_2sm(void* dst, const CUtensorMap* m, uint32_t mbar_cluster, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(mbar_cluster), "r"(x), "r"(y), "r"(z) : "memory");
}
__device__ __forceinline__ void tma2_2sm(void* dst, const CUtensorMap* m, uint32_t mbar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
          "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(m)), "r"(mbar_cluster), "r"(x), "r"(y) : "memory");
}
// Bring a weight tile into L2 ahead of its shared-memory load (no completion to wait for).
__device__ __forceinline__ void pf_l2(const CUtensorMap* m, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y) : "memory");
}
// Advance a shared-memory descriptor by `units` x 16 bytes: the start-address field is
// the low 14 bits, and no shared-memory address reaches 2^18 bytes, so the add never
// carries out of the field.
__device__ __forceinline__ uint64_t desc_advance(uint64_t d, uint32_t units) {
  uint32_t lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(d));
  lo += units;
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void umma2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
               "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void umma2_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\ttcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
               "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc) : "memory");
}
// Instruction descriptor of kind::f8f6f4 with e4m3 A and B (format code 0) and fp32 D.
__host__ __device__ constexpr uint32_t make_idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Packed fp32x2 arithmetic (one instruction for two lanes of a row).
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ float2 acc2(const uint32_t (&v)[32], int i) {
  return make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Dequantised accumulator columns: acc * a_scale(row) * w_scale(col), in place.
struct Dequant {
  float as;          // this row's activation scale (1 when not quantised)
  const float* ws;   // column scales of the tile (null when not quantised)
};
__device__ __forceinline__ void dequant32(uint32_t (&v)[32], const Dequant& dq, int col) {
  if (!dq.ws) return;
  const float4* w4 = reinterpret_cast<const float4*>(dq.ws + col);
  const float2 as2 = f2(dq.as, dq.as);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 w = __ldg(w4 + i);
    const float2 a = __fmul2_rn(__fmul2_rn(acc2(v, 2 * i), as2), f2(w.x, w.y));
    const float2 b = __fmul2_rn(__fmul2_rn(acc2(v, 2 * i + 1), as2), f2(w.z, w.w));
    v[4 * i + 0] = __float_as_uint(a.x);
    v[4 * i + 1] = __float_as_uint(a.y);
    v[4 * i + 2] = __float_as_uint(b.x);
    v[4 * i + 3] = __float_as_uint(b.y);
  }
}

__device__ __forceinline__ void commit_both(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "h"((uint16_t)3) : "memory");
}

__device__ __forceinline__ void store_row32(bf16* dst, const float* f) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d[i] = make_uint4(pack_bf16x2(f[8 * i + 0], f[8 * i + 1]), pack_bf16x2(f[8 * i + 2], f[8 * i + 3]),
                      pack_bf16x2(f[8 * i + 4], f[8 * i + 5]), pack_bf16x2(f[8 * i + 6], f[8 * i + 7]));
}

__device__ __forceinline__ void load_row32(const bf16* src, float* f) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = s[i];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 v = unpack_bf16x2(w[j]);
      f[8 * i + 2 * j] = v.x;
      f[8 * i + 2 * j + 1] = v.y;
    }
  }
}

__device__ __forceinline__ void store_row32_f32(float* dst, const float* f) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 8; ++i) d[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
}

__device__ __forceinline__ void load_row32_f32(const float* src, float* f) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = s4[i];
    f[4 * i] = v.x;
    f[4 * i + 1] = v.y;
    f[4 * i + 2] = v.z;
    f[4 * i + 3] = v.w;
  }
}

// SwiGLU over one packed 256-column accumulator: 128 outputs at dst[0..128).
// silu(g) = g / (1 + 2^(-g log2 e)) with MUFU ex2 and rcp.approx.
// Chunks [c_begin, c_end) of the 4 (one epilogue warp takes two).
__device__ __forceinline__ void epi_swiglu(uint32_t tbase, bool row_ok, bf16* dst, int cols_left, const Dequant& dq,
                                           int col0, int c_begin, int c_end) {
  const float2 nl2e = f2(-1.4426950408889634f, -1.4426950408889634f), one = f2(1.0f, 1.0f);
#pragma unroll 1
  for (int c = c_begin; c < c_end; ++c) {
    uint32_t g[32], u[32];
    tmem_load32(tbase + c * 32, g);
    tmem_load32(tbase + 128 + c * 32, u);
    dequant32(g, dq, col0 + c * 32);
    dequant32(u, dq, col0 + 128 + c * 32);
    if (row_ok && c * 32 < cols_left) {
      float o[32];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 gg = acc2(g, i);
        float2 t = __fmul2_rn(gg, nl2e);
        t = __fadd2_rn(f2(ex2_approx(t.x), ex2_approx(t.y)), one);
        const float2 r = __fmul2_rn(__fmul2_rn(gg, f2(rcp_approx(t.x), rcp_approx(t.y))), acc2(u, i));
        o[2 * i] = r.x;
        o[2 * i + 1] = r.y;
      }
      store_row32(dst + c * 32, o);
    }
  }
}

// One 128-column head of the QKV projection: V stored as is; Q and K get RMSNorm over the
// head (fp32, eps) times the learned weight, then RoPE on adjacent pairs from the table.
__device__ __forceinline__ void epi_qkv_head(uint32_t tb, bool row_ok, int which, bf16* dst, const bf16* nw,
                                             const float* rope_row, float eps, const Dequant& dq, int col0) {
  if (which == 2) {
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t v[32];
      tmem_load32(tb + c * 32, v);
      dequant32(v, dq, col0 + c * 32);
      if (row_ok) {
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]);
        store_row32(dst + c * 32, o);
      }
    }
    return;
  }
  float2 ss2 = f2(0.f, 0.f);
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t v[32];
    tmem_load32(tb + c * 32, v);
    dequant32(v, dq, col0 + c * 32);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 x = acc2(v, i);
      ss2 = __ffma2_rn(x, x, ss2);
    }
  }
  const float rs = rsqrtf((ss2.x + ss2.y) * (1.0f / 128.0f) + eps);
  const float2 rs2 = f2(rs, rs);
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t v[32];
    tmem_load32(tb + c * 32, v);
    dequant32(v, dq, col0 + c * 32);
    if (row_ok) {
      float w[32];
      load_row32(nw + c * 32, w);  // 16-byte loads of the norm weights
      float o[32];
      const float4* rp = reinterpret_cast<const float4*>(rope_row + c * 32);  // 16 pairs (cos, sin)
#pragma unroll
      for (int p = 0; p < 16; p += 2) {
        const float4 cs = __ldg(rp + p / 2);  // pair p: (cs.x, cs.y), pair p+1: (cs.z, cs.w)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int d = 2 * (p + h);
          const float co = h ? cs.z : cs.x, si = h ? cs.w : cs.y;
          const float2 x = __fmul2_rn(__fmul2_rn(acc2(v, p + h), rs2), f2(w[d], w[d + 1]));
          // (x0 c - x1 s, x1 c + x0 s)
          const float2 r = __ffma2_rn(x, f2(co, co), __fmul2_rn(f2(x.y, x.x), f2(-si, si)));
          o[d] = r.x;
          o[d + 1] = r.y;
        }
      }
      store_row32(dst + c * 32, o);
    }
  }
}

// kFp8: A and W are e4m3 (k-blocks of 128 elements, still 128-byte rows; kind::f8f6f4,
// K 32 per MMA); the epilogue dequantises with the per-row and per-column scales.
template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmParams P) {
  constexpr int KB = kFp8 ? 128 : BK;  // elements per k-block
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kATileBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank();          // 0 = leader (issues the MMAs), 1 = peer
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], 16);  // 8 epilogue warps in each CTA of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < P.nprob; ++p) {
      tma_prefetch_desc(&P.a_map[p]);
      tma_prefetch_desc(&P.b_map[p]);
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{P.status, abort_flag, kWaitLimitNs};
  grid_dependency_wait();  // A, residuals and outputs belong to earlier kernels of the stream
  allow_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int t = pair; t < P.total_tiles && ok; t += npairs) {
        const TileInfo ti = decode_tile(P, t);
        const DevProblem& pr = P.prob[ti.p];
        const int kblocks = (pr.k + KB - 1) / KB;
        const int arow = pr.a_row0 + ti.m_tile * PAIR_M + (int)rank * BM;
        const int brow = ti.n_tile * BN + (int)rank * (BN / 2);
        const bool pf = ti.m_tile == 0;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (pf && kb + 8 < kblocks) pf_l2(&P.b_map[ti.p], (kb + 8) * KB, brow);
          if (!mbar_wait_sleep(&empty[stage], phase ^ 1u, wc, kSiteEmpty)) {
            ok = false;
            break;
          }
          // both CTAs' loads complete on the leader's full barrier
          const uint32_t fb = map_to_rank(smem_u32(&full[stage]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * kStageBytes);
          tma3_2sm(sA + stage * kATileBytes, &P.a_map[ti.p], fb, kb * KB, arow, ti.b);
          tma2_2sm(sB + stage * kBTileBytes, &P.b_map[ti.p], fb, kb * KB, brow);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && rank == 0) {
        const long long outstanding = issued < kStages ? issued : kStages;
        for (long long i = 0; i < outstanding; ++i) {
          if (stage == 0) {
            stage = kStages;
            phase ^= 1u;
          }
          --stage;
          const uint64_t t0 = global_timer_ns();
          while (!mbar_try(&full[stage], phase) && global_timer_ns() - t0 < 100000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (lane == 0 && rank == 0) {
      const uint32_t idesc = kFp8 ? make_idesc_e4m3(PAIR_M, BN) : make_idesc_bf16(PAIR_M, BN, false);
      const uint64_t a_desc0 = make_sdesc_sw128(smem_u32(sA), 16, 1024);
      const uint64_t b_desc0 = make_sdesc_sw128(smem_u32(sB), 16, 1024);
      uint32_t stage = 0, phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = pair; t < P.total_tiles && ok; t += npairs, ++local) {
        const TileInfo ti = decode_tile(P, t);
        const DevProblem& pr = P.prob[ti.p];
        const int kblocks = (pr.k + KB - 1) / KB;
        const int acc = local & 1;
        if (!mbar_wait(&acc_empty[acc], ((uint32_t)(local >> 1) & 1u) ^ 1u, wc, kSiteAccEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, wc, kSiteFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = desc_advance(a_desc0, stage * (kATileBytes >> 4));
          const uint64_t bd = desc_advance(b_desc0, stage * (kBTileBytes >> 4));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // 32 bytes of K per MMA: 16 bf16 or 32 e4m3
            if (kFp8)
              umma2_f8(d_tmem, desc_advance(ad, kk * 2), desc_advance(bd, kk * 2), idesc, (kb | kk) != 0 ? 1u : 0u);
            else
              umma2(d_tmem, desc_advance(ad, kk * 2), desc_advance(bd, kk * 2), idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          commit_both(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        commit_both(&acc_full[acc]);
      }
      asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(drain))
                   : "memory");
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try(drain, 0) && global_timer_ns() - t0 < 1000000000ull) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int eh = (warp - 2) >> 2;  // the 128-column half of the accumulator this warp takes
    const uint32_t acc_empty_leader0 = map_to_rank(smem_u32(&acc_empty[0]), 0);
    const uint32_t acc_empty_leader1 = map_to_rank(smem_u32(&acc_empty[1]), 0);
    int local = 0;
    for (int t = pair; t < P.total_tiles; t += npairs, ++local) {
      const int acc = local & 1;
      bool ok = mbar_wait_sleep(&acc_full[acc], (uint32_t)(local >> 1) & 1u, wc, kSiteAccFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const TileInfo ti = decode_tile(P, t);
      const DevProblem& pr = P.prob[ti.p];
      const uint32_t tbase = tmem + (uint32_t)(acc * BN) + ((uint32_t)(q * 32) << 16);
      const int r = ti.m_tile * PAIR_M + (int)rank * BM + q * 32 + lane;
      const bool row_ok = r < pr.rows;
      const int col0 = ti.n_tile * BN;
      Dequant dq{1.0f, nullptr};
      if (kFp8) {
        dq.as = row_ok ? pr.a_scale[(long long)ti.b * pr.a_rows_total + pr.a_row0 + r] : 0.f;
        dq.ws = pr.w_scale;
      }
      if (pr.epi == kEpiStore || pr.epi == kEpiResidual) {
        const long long off = (long long)ti.b * pr.out_bstride + (long long)(pr.out_row0 + r) * pr.ld_out +
                              pr.out_col0 + col0;
        const bf16* grow = pr.gate ? pr.gate + (long long)ti.b * pr.gate_stride + col0 : nullptr;
        const float gsc = pr.coef ? pr.coef[ti.b] : 0.f;
#pragma unroll 1
        for (int c = eh * 4; c < eh * 4 + 4; ++c) {
          uint32_t v[32];
          tmem_load32(tbase + c * 32, v);
          if (kFp8 && col0 + c * 32 < pr.n) dequant32(v, dq, col0 + c * 32);
          if (row_ok && col0 + c * 32 < pr.n) {
            float o[32];
            if (pr.epi == kEpiResidual) {
              float xr[32];
              if (pr.res_f32) load_row32_f32(pr.res_f32 + off + c * 32, xr);
              else load_row32(pr.res + off + c * 32, xr);
              if (pr.coef) {
                const float2 g2 = f2(gsc, gsc);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float2 r = __ffma2_rn(g2, acc2(v, i), f2(xr[2 * i], xr[2 * i + 1]));
                  o[2 * i] = r.x;
                  o[2 * i + 1] = r.y;
                }
              } else {
                float gv[32];
                load_row32(grow + c * 32, gv);  // 16-byte loads of the gate vector
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float2 r = __ffma2_rn(f2(gv[2 * i], gv[2 * i + 1]), acc2(v, i), f2(xr[2 * i], xr[2 * i + 1]));
                  o[2 * i] = r.x;
                  o[2 * i + 1] = r.y;
                }
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]);
            }
            if (pr.out_f32) store_row32_f32(pr.out_f32 + off + c * 32, o);
            if (pr.out) store_row32(pr.out + off + c * 32, o);
          }
        }
      } else if (pr.epi == kEpiSwiGLU || (pr.epi == kEpiQKV && col0 >= pr.n_qkv)) {
        const int ocol = (col0 - (pr.epi == kEpiQKV ? pr.n_qkv : 0)) / 2;
        const int n_out = (pr.n - (pr.epi == kEpiQKV ? pr.n_qkv : 0)) / 2;
        bf16* orow = pr.out + (long long)ti.b * pr.out_bstride + (long long)(pr.out_row0 + r) * pr.ld_out +
                     pr.out_col0 + ocol;
        epi_swiglu(tbase, row_ok, orow, n_out - ocol, dq, col0, 2 * eh, 2 * eh + 2);
      } else {
        const int which = col0 / pr.hidden;
        const int heads = pr.hidden / 128;
        const int tok = pr.tok0 + r;
        bf16* base = which == 0 ? pr.q : (which == 1 ? pr.kk : pr.v);
        const bf16* nw = which == 0 ? pr.q_norm : pr.k_norm;
        const float* rope_row = pr.rope + (long long)(row_ok ? tok : 0) * 128;
#pragma unroll 1
        for (int hh = eh; hh < eh + 1; ++hh) {
          const int head = (col0 % pr.hidden) / 128 + hh;
          bf16* dst = base + (((long long)ti.b * heads + head) * pr.seq + tok) * 128;
          epi_qkv_head(tbase + hh * 128, row_ok, which, dst, nw, rope_row, P.eps, dq, col0 + hh * 128);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_cluster(acc ? acc_empty_leader1 : acc_empty_leader0);
    }
  }

  tc_fence_before();
  cluster_sync_all();  // no MMA, TMA or remote arrive of the pair is still in flight
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// the shared-memory attribute has been raised for (device, operand type) (any host thread)
std::atomic<bool> g_attr_set[32];

}  // namespace

cudaError_t launch_gemm(const GemmProblemHost* probs, int nprob, int batch, float eps, DeviceStatus* status,
                        int cls, cudaStream_t s) {
  if (nprob < 1 || nprob > 2) return cudaErrorInvalidValue;
  GemmParams P;
  memset(&P, 0, sizeof(P));
  int tiles = 0;
  for (int i = 0; i < nprob; ++i) {
    const GemmProblemHost& h = probs[i];
    DevProblem& d = P.prob[i];
    if (h.rows <= 0 || h.n <= 0 || h.k <= 0 || !h.a || !h.w) return cudaErrorInvalidValue;
    // every pointer the chosen epilogue dereferences must be present
    switch (h.epi) {
      case kEpiStore:
        if (!h.out) return cudaErrorInvalidValue;
        break;
      case kEpiResidual:
        if ((!h.gate && !h.coef) || (!h.out && !h.out_f32) || (!h.res && !h.res_f32 && !h.out))
          return cudaErrorInvalidValue;
        break;
      case kEpiSwiGLU:
        if (!h.out) return cudaErrorInvalidValue;
        break;
      case kEpiQKV:
        if (!h.q || !h.kk || !h.v || !h.q_norm || !h.k_norm || !h.rope || h.hidden <= 0 ||
            (h.n > h.n_qkv && !h.out))
          return cudaErrorInvalidValue;
        break;
      default:
        return cudaErrorInvalidValue;
    }
    const int esz = h.fp8 ? 1 : 2;
    if (h.fp8 != probs[0].fp8) return cudaErrorInvalidValue;
    if (h.fp8 && (!h.a_scale || !h.w_scale || (h.k % 16) != 0)) return cudaErrorInvalidValue;
    const uint64_t adims[3] = {(uint64_t)h.k, (uint64_t)h.a_rows_total, (uint64_t)batch};
    const uint64_t astr[2] = {(uint64_t)h.lda * esz, (uint64_t)h.lda * esz * (uint64_t)h.a_rows_total};
    const uint32_t kbx = h.fp8 ? 128 : BK;
    const uint32_t abox[3] = {kbx, BM, 1};
    const uint64_t bdims[2] = {(uint64_t)h.k, (uint64_t)h.n};
    const uint64_t bstr[1] = {(uint64_t)h.k * esz};
    const uint32_t bbox[2] = {kbx, BN / 2};
    if (h.fp8) {
      if (!encode_tmap_u8(&P.a_map[i], h.a, 3, adims, astr, abox)) return cudaErrorInvalidValue;
      if (!encode_tmap_u8(&P.b_map[i], h.w, 2, bdims, bstr, bbox)) return cudaErrorInvalidValue;
    } else {
      if (!encode_tmap_bf16(&P.a_map[i], h.a, 3, adims, astr, abox)) return cudaErrorInvalidValue;
      if (!encode_tmap_bf16(&P.b_map[i], h.w, 2, bdims, bstr, bbox)) return cudaErrorInvalidValue;
    }
    d.rows = h.rows;
    d.a_row0 = h.a_row0;
    d.n = h.n;
    d.k = h.k;
    d.m_tiles = (h.rows + PAIR_M - 1) / PAIR_M;
    d.n_tiles = (h.n + BN - 1) / BN;
    d.tile_begin = tiles;
    d.epi = h.epi;
    d.out = h.out;
    d.out_f32 = h.out_f32;
    d.res = h.res;
    d.res_f32 = h.res_f32;
    if (h.epi == kEpiResidual && !h.res && !h.res_f32) d.res = h.out;
    d.out_bstride = h.out_bstride;
    d.ld_out = h.ld_out;
    d.out_row0 = h.out_row0;
    d.out_col0 = h.out_col0;
    d.gate = h.gate;
    d.gate_stride = h.gate_stride;
    d.coef = h.coef;
    d.a_scale = h.a_scale;
    d.w_scale = h.w_scale;
    d.a_rows_total = h.a_rows_total;
    d.n_qkv = h.n_qkv;
    d.hidden = h.hidden;
    d.q = h.q;
    d.kk = h.kk;
    d.v = h.v;
    d.q_norm = h.q_norm;
    d.k_norm = h.k_norm;
    d.rope = h.rope;
    d.seq = h.seq;
    d.tok0 = h.tok0;
    tiles += d.m_tiles * d.n_tiles * batch;
  }
  P.nprob = nprob;
  P.batch = batch;
  P.total_tiles = tiles;
  P.eps = eps;
  P.status = status;
  if (tiles == 0) return cudaSuccess;

  int dev = 0;
  cudaGetDevice(&dev);
  const bool fp8 = probs[0].fp8 != 0;
  const int slot = dev * 2 + (fp8 ? 1 : 0);
  if (dev < 16 && !g_attr_set[slot].load(std::memory_order_acquire)) {
    cudaError_t e = fp8 ? cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kSmemBytes)
                        : cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    g_attr_set[slot].store(true, std::memory_order_release);
  }
  const int pairs_max = sm_count() / 2;
  const int pairs = tiles < pairs_max ? tiles : pairs_max;
  LaunchScope scope(cls, s);
  if (fp8) return launch_k(gemm_kernel<true>, dim3(2 * pairs), dim3(kThreads), kSmemBytes, s, P);
  return launch_k(gemm_kernel<false>, dim3(2 * pairs), dim3(kThreads), kSmemBytes, s, P);
}

}  // namespace dit
