// Joint text + image attention on the tensor cores: O = softmax(Q K^T / sqrt(128)) V over
// every key of the joint sequence, no mask ("flux2-klein-p100a" Caveats: all 512 padded
// text rows enter with no mask; reading R6 for the scale).  Padded tail keys of a tile
// (sequence length not a multiple of 128) are masked out, padded tail queries not stored.
//
// One CTA per (pair of 128-query tiles, head, batch row), 320 threads:
//   warp 0      TMA: Q0, Q1 and K_0 once; then per key block j one ring slot (two slots)
//               holding V_j and K_{j+1} (128 keys x 128 dims as two 64-dim halves, 128-byte
//               swizzle) behind a single barrier, so that the MMA thread waits once per block;
//   warp 1      tcgen05.mma from one thread, in the order
//                 S0 = Q0 K_0^T, S1 = Q1 K_0^T, then for every key block j:
//                 O0 += P0 V_j, S0 = Q0 K_{j+1}^T, O1 += P1 V_j, S1 = Q1 K_{j+1}^T,
//               so that one tile's softmax overlaps the other tile's MMAs.  Its only
//               commits are the two "S_t ready" signals per block: a ring slot is released
//               by a softmax thread of tile 1 once it sees S1 of the next block (every MMA
//               reading the slot was issued before it), which saves the issuer a commit per
//               slot -- on sm_103a an issuing thread is held ~one MMA time per commit;
//   warps 2-5   softmax of tile 0, warps 6-9 softmax of tile 1: one thread per query row,
//               S row streamed from TMEM in 32-key chunks, exp2 against the running
//               maximum with log2(e)/sqrt(d) folded in, P rounded to bf16 and written back
//               into TMEM over its own S, where the PV MMA reads it as its A operand.  The
//               running maximum is lazy: the exponentials of a key block are taken against
//               the maximum so far, and only when the block's row sum of P passes 2^12 (some
//               key exceeded the maximum by more than 12 in log2 units) are the block
//               maximum, the rescale of O (in TMEM) and the exponentials redone; the result is
//               exact after the final 1/l.  Only then (and on the first key block) is S read
//               twice, and the common path computes no maximum at all.
// Why the common path avoids 3-input max and scalar FP32 arithmetic: on sm_103a a warp that
// issues tcgen05.mma competes for issue slots with the other warps of its SM sub-partition,
// and dense scalar FMA / max / byte-permute streams there slow the MMA issue several-fold
// (measured: 64 -> 88 cycles per M128 N128 K16 MMA under dense 3-input max, -> 340 under
// dense scalar FMA), while packed fp32x2 FMA/add, MUFU ex2 and bf16x2 conversion do not.
// The MMA thread issues from descriptors computed once, and the TMA warp and the output
// waits sleep on their barriers instead of spinning, for the same reason.  The softmax warps
// spin on "S ready": waking from a sleeping wait added a few hundred cycles to every key
// block (about 1 % of the kernel).
// Output: each tile's O / l is staged as bf16 in that tile's (then free) Q shared memory, in
// the 128-byte-swizzled layout the Q loads used, and written by TMA stores through a 3-D
// view of the output, which clips the rows of a partial last tile.
// Ordering: MMAs issued by one thread execute in order and a commit tracks every earlier
// MMA of that thread, so "S_t of block j+1 is ready" also means "P_t V_j is complete":
// the softmax may then rescale O_t and overwrite P_t without a further wait.
// TMEM (512 columns): tile t uses S_t / P_t at [256t, 256t + 128) and O_t at
// [256t + 128, 256t + 256).
#include <math.h>

#include <atomic>

#include "runtime.h"

namespace dit {

namespace {

constexpr int kBQ = 128, kBKV = 128;
constexpr int kThreads = 320;
constexpr uint32_t kHalfBytes = 128 * 64 * 2;   // one 64-dim half of a 128-row tile
constexpr uint32_t kTileBytes = 2 * kHalfBytes;  // 32 KB
constexpr uint32_t kOffQ = 0;                    // Q0, Q1
constexpr uint32_t kOffK = kOffQ + 2 * kTileBytes;
constexpr uint32_t kOffV = kOffK + 2 * kTileBytes;
constexpr uint32_t kOffBar = kOffV + 2 * kTileBytes;
constexpr size_t kSmemBytes = 1024 + kOffBar + 256;
constexpr uint32_t kTmemCols = 512;
constexpr float kPsumLimit = 4096.0f;  // row sum of P that sends a key block down the slow path

struct alignas(64) AttnParams {
  CUtensorMap q_map, k_map, v_map;
  CUtensorMap o_map;  // output [B][n][ld_out] viewed 3-D, stored by TMA from the Q tiles' smem
  bf16* out;
  int ld_out, n, heads;
  float scale_log2;
  DeviceStatus* status;
};

// ---- softmax arithmetic helpers -----------------------------------------------------

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (d0, d1) = (a0, a1) * b + c with one packed fp32x2 FMA.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  uint64_t A, B, C, D;
  asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(B) : "f"(b));
  asm("mov.b64 %0, {%1, %1};" : "=l"(C) : "f"(c));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(D) : "l"(A), "l"(B), "l"(C));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(D));
}

// (s0, s1) += (a0, a1) with one packed fp32x2 add.
__device__ __forceinline__ void fadd2(float& s0, float& s1, float a0, float a1) {
  uint64_t S, A;
  asm("mov.b64 %0, {%1, %2};" : "=l"(S) : "f"(s0), "f"(s1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(A) : "f"(a0), "f"(a1));
  asm("add.f32x2 %0, %0, %1;" : "+l"(S) : "l"(A));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(s0), "=f"(s1) : "l"(S));
}

// One 32-key chunk of a softmax row: P = 2^(s c - m) packed to bf16 pairs and the two
// partial row sums; kMax: also the running key maximum (raw scores); kTail: keys at or past
// kv_valid masked to -inf.  Every exponential runs on MUFU: moving a share of them to an
// FMA-pipe polynomial was measured slower here.
template <bool kTail, bool kMax>
__device__ __forceinline__ void softmax_chunk(const uint32_t (&r)[32], int base, int kv_valid, float c, float mneg,
                                              float& smax, float& ps0, float& ps1, uint32_t* pk) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    float s0 = __uint_as_float(r[i]), s1 = __uint_as_float(r[i + 1]);
    if (kTail) {
      if (base + i >= kv_valid) s0 = -INFINITY;
      if (base + i + 1 >= kv_valid) s1 = -INFINITY;
    }
    if (kMax) smax = fmax3(smax, s0, s1);
    float x0, x1;
    ffma2(x0, x1, s0, s1, c, mneg);
    const float p0 = ex2_approx(x0);
    const float p1 = ex2_approx(x1);
    fadd2(ps0, ps1, p0, p1);
    pk[i / 2] = pack_bf16x2(p0, p1);
  }
}

template <bool kTail, bool kMax>
__device__ __forceinline__ void softmax_row(uint32_t tS, int kv_valid, float c, float mneg, float& smax, float& psum,
                                            uint32_t (&pk)[64]) {
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t r[32];
    tmem_load32(tS + q * 32, r);
    softmax_chunk<kTail, kMax>(r, q * 32, kv_valid, c, mneg, smax, ps0, ps1, &pk[q * 16]);
  }
  psum = ps0 + ps1;
}

enum : uint32_t { kSiteQ = 0x201, kSiteFree, kSiteReady, kSitePFull, kSiteSFull, kSiteODone, kSiteOSync };

// Store a {64, 128, 1} box of the output from shared memory (128-byte swizzle, the layout
// of a Q half-tile); rows past the tensor's end are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_store_commit_and_drain() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // smem read out: safe to exit
}


// Shared-memory descriptors of every MMA operand, computed once: Q_t (A of S_t = Q_t K^T),
// K and V of both ring stages (B operands), per 16-wide K step.
struct Descs {
  uint64_t q[2][8], k[2][8], v[2][8];
};

__device__ __forceinline__ void make_descs(uint8_t* smem, Descs& d) {
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
      d.q[t][kk] = make_sdesc_sw128(smem_u32(smem + kOffQ + t * kTileBytes) + off, 16, 1024);
      d.k[t][kk] = make_sdesc_sw128(smem_u32(smem + kOffK + t * kTileBytes) + off, 16, 1024);
      d.v[t][kk] = make_sdesc_sw128(smem_u32(smem + kOffV + t * kTileBytes) + kk * 2048, kHalfBytes, 1024);
    }
}

// Eight back-to-back MMAs (K = 128) from one asm statement: D = A B (first) then D += A B.
__device__ __forceinline__ void umma8_ss(uint32_t d, const uint64_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t"
      "setp.ne.b32 pf, %18, %18;\n\t"
      "setp.eq.b32 pt, %18, %18;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %17, pf;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %17, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %17, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %17, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %17, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %17, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %17, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %17, pt;\n\t}" ::"r"(d),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]), "l"(b[1]),
      "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc), "r"(0)
      : "memory");
}

// Eight MMAs with A read from TMEM at columns a_tmem + 8 kk: D (+)= A B.
__device__ __forceinline__ void umma8_ts(uint32_t d, uint32_t a_tmem, const uint64_t (&b)[8], uint32_t idesc,
                                         uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred pa, pt;\n\t.reg .b32 t1, t2, t3, t4, t5, t6, t7;\n\t"
      "setp.ne.b32 pa, %11, 0;\n\t"
      "setp.eq.b32 pt, %11, %11;\n\t"
      "add.u32 t1, %1, 8;\n\tadd.u32 t2, %1, 16;\n\tadd.u32 t3, %1, 24;\n\tadd.u32 t4, %1, 32;\n\t"
      "add.u32 t5, %1, 40;\n\tadd.u32 t6, %1, 48;\n\tadd.u32 t7, %1, 56;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %10, pa;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t1], %3, %10, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t2], %4, %10, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t3], %5, %10, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t4], %6, %10, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t5], %7, %10, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t6], %8, %10, pt;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [t7], %9, %10, pt;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc),
      "r"(acc)
      : "memory");
}

// S_t = Q_t K^T (K from ring stage ST), then arrive on `bar` when done.
template <int ST>
__device__ __forceinline__ void issue_qk(const Descs& d, uint32_t tmem, int t, uint32_t idesc, uint64_t* bar) {
  umma8_ss(tmem + (uint32_t)(t * 256), d.q[t], d.k[ST], idesc);
  umma_commit(bar);
}

// O_t (+)= P_t V (V from ring stage ST), P_t read from TMEM over S_t.
template <int ST>
__device__ __forceinline__ void issue_pv(const Descs& d, uint32_t tmem, int t, bool acc, uint32_t idesc) {
  umma8_ts(tmem + (uint32_t)(t * 256 + 128), tmem + (uint32_t)(t * 256), d.v[ST], idesc, acc ? 1u : 0u);
}

// One key block j (ring stage ST = j & 1) of the MMA issuer, once V_j and K_{j+1} have
// landed (one barrier for both):
//   O0 += P0 V_j, S0 = Q0 K_{j+1}^T, O1 += P1 V_j, S1 = Q1 K_{j+1}^T.
template <int ST>
__device__ __forceinline__ bool mma_block(const Descs& d, uint32_t tmem, int j, int nkv, uint32_t idesc_qk,
                                          uint32_t idesc_pv, uint64_t* ready, uint64_t* s_full, uint64_t* p_full,
                                          uint64_t* o_done, const WaitCtx& wc) {
  constexpr int NST = ST ^ 1;
  const bool more = j + 1 < nkv;
  if (!mbar_wait(&ready[ST], (uint32_t)(j >> 1) & 1u, wc, kSiteReady) ||
      !mbar_wait(&p_full[0], (uint32_t)j & 1u, wc, kSitePFull))
    return false;
  tc_fence_after();
  issue_pv<ST>(d, tmem, 0, j > 0, idesc_pv);
  if (more)
    issue_qk<NST>(d, tmem, 0, idesc_qk, &s_full[0]);
  else
    umma_commit(&o_done[0]);  // tile 0's output may be read while tile 1 finishes
  if (!mbar_wait(&p_full[1], (uint32_t)j & 1u, wc, kSitePFull)) return false;
  tc_fence_after();
  issue_pv<ST>(d, tmem, 1, j > 0, idesc_pv);
  if (more)
    issue_qk<NST>(d, tmem, 1, idesc_qk, &s_full[1]);
  else
    umma_commit(&o_done[1]);
  return true;
}

__global__ void __launch_bounds__(kThreads, 1) attention_kernel(const __grid_constant__ AttnParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* q_full = bars + 0;   // Q0, Q1 and K_0
  uint64_t* ready = bars + 1;    // [2] ring slot: V_j and K_{j+1} landed
  uint64_t* slot_free = bars + 3;  // [2] ring slot: every MMA reading V_j and K_{j+1} done
  uint64_t* s_full = bars + 5;   // [2] per tile
  uint64_t* p_full = bars + 7;   // [2] per tile
  uint64_t* o_done = bars + 9;   // [2] per tile: its last PV MMA is done
  uint64_t* drain = bars + 11;
  uint64_t* osync = bars + 12;   // [2] per tile: its 4 warps have staged the output
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = P.n;
  const int nkv = (n + kBKV - 1) / kBKV;
  const int q0 = blockIdx.x * (2 * kBQ);
  const int head = blockIdx.y, b = blockIdx.z;
  const int bh = b * P.heads + head;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ready[i], 1);
      mbar_init(&slot_free[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_done[i], 1);
      mbar_init(&osync[i], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&P.q_map);
    tma_prefetch_desc(&P.k_map);
    tma_prefetch_desc(&P.v_map);
    tma_prefetch_desc(&P.o_map);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{P.status, abort_flag, kWaitLimitNs};
  grid_dependency_wait();  // Q, K, V and the output belong to earlier kernels of the stream
  allow_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Ring slot b = j & 1 carries V_j (V stage b) and K_{j+1} (K stage (j+1) & 1).  Slot
    // j (j >= 1) is loaded once S1 of block j - 1 is complete: that ends every read of the
    // V_{j-2} and K_{j-1} it overwrites (for j = 1, of K_0 by the first two MMAs).
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(q_full, 3 * kTileBytes);
      for (int t = 0; t < 2; ++t) {
        tma_load_3d(smem + kOffQ + t * kTileBytes, &P.q_map, q_full, 0, q0 + t * kBQ, bh);
        tma_load_3d(smem + kOffQ + t * kTileBytes + kHalfBytes, &P.q_map, q_full, 64, q0 + t * kBQ, bh);
      }
      tma_load_3d(smem + kOffK, &P.k_map, q_full, 0, 0, bh);
      tma_load_3d(smem + kOffK + kHalfBytes, &P.k_map, q_full, 64, 0, bh);
      for (int j = 0; j < nkv; ++j) {
        const int b = j & 1;
        if (j >= 1 && !mbar_wait_sleep(&slot_free[b], (uint32_t)((j - 1) >> 1) & 1u, wc, kSiteFree)) {
          ok = false;
          break;
        }
        const bool k_next = j + 1 < nkv;
        mbar_arrive_expect_tx(&ready[b], k_next ? 2 * kTileBytes : kTileBytes);
        tma_load_3d(smem + kOffV + b * kTileBytes, &P.v_map, &ready[b], 0, j * kBKV, bh);
        tma_load_3d(smem + kOffV + b * kTileBytes + kHalfBytes, &P.v_map, &ready[b], 64, j * kBKV, bh);
        if (k_next) {
          const int kb = (j + 1) & 1;
          tma_load_3d(smem + kOffK + kb * kTileBytes, &P.k_map, &ready[b], 0, (j + 1) * kBKV, bh);
          tma_load_3d(smem + kOffK + kb * kTileBytes + kHalfBytes, &P.k_map, &ready[b], 64, (j + 1) * kBKV, bh);
        }
        issued = j + 1;
      }
      if (!ok) {
        // Unwinding: let copies in flight land (bounded) before the block exits.
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try(q_full, 0) && global_timer_ns() - t0 < 100000000ull) {
        }
        for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
          while (!mbar_try(&ready[j & 1], (uint32_t)(j >> 1) & 1u) && global_timer_ns() - t0 < 200000000ull) {
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc_bf16(128, 128, false);
      const uint32_t idesc_pv = make_idesc_bf16(128, 128, true);
      Descs d;
      make_descs(smem, d);
      bool ok = mbar_wait(q_full, 0, wc, kSiteQ);
      if (ok) {
        tc_fence_after();
        issue_qk<0>(d, tmem, 0, idesc_qk, &s_full[0]);
        issue_qk<0>(d, tmem, 1, idesc_qk, &s_full[1]);
      }
      for (int j = 0; j < nkv && ok; j += 2) {
        ok = mma_block<0>(d, tmem, j, nkv, idesc_qk, idesc_pv, ready, s_full, p_full, o_done, wc);
        if (ok && j + 1 < nkv)
          ok = mma_block<1>(d, tmem, j + 1, nkv, idesc_qk, idesc_pv, ready, s_full, p_full, o_done, wc);
      }
      umma_commit(drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_try(drain, 0) && global_timer_ns() - t0 < 1000000000ull) {
      }
    }
  } else {
    // ------------------------------------------------------------ softmax / correction / output
    const int tile = (warp - 2) >> 2;  // warps 2-5 -> tile 0, warps 6-9 -> tile 1
    const int qq = warp & 3;           // TMEM lane quarter of this warp
    const int row = qq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const uint32_t tS = tmem + (uint32_t)(tile * 256) + lane_off;
    const uint32_t tO = tS + 128;
    const float c = P.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      ok = mbar_wait(&s_full[tile], (uint32_t)j & 1u, wc, kSiteSFull);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // S1 of block j is complete, hence every MMA issued before it: the reads of V_{j-1}
      // (V stage (j+1) & 1) and of K_j (K stage j & 1) are done, which is what the
      // slot of key block j + 1 (V_{j+1}, K_{j+2}) overwrites.
      if (tile == 1 && qq == 2 && lane == 0) mbar_arrive(&slot_free[(j + 1) & 1]);
      tc_fence_after();
      const int kv_valid = n - j * kBKV;
      // Fast path: exponentials against the running maximum, streamed over four
      // 32-key chunks of S, only the packed P kept.  Valid while the row sum of P stays
      // at or below kPsumLimit (no key far above the running maximum); never on the first
      // key block, which has no maximum yet.  NaN scores keep the fast path.
      uint32_t pk[64];
      float psum = 0.f, smax = -INFINITY;
      bool slow = (j == 0);
      if (!slow) {
        if (kv_valid >= kBKV)
          softmax_row<false, false>(tS, kv_valid, c, -m_run, smax, psum, pk);
        else
          softmax_row<true, false>(tS, kv_valid, c, -m_run, smax, psum, pk);
        slow = psum > kPsumLimit;
      }
      float alpha = 1.0f;
      if (__any_sync(0xffffffffu, slow)) {
        // Slow path (whole warp): the block maximum first, then the exponentials again.
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t r[32];
          tmem_load32(tS + q * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (kv_valid >= kBKV || q * 32 + i < kv_valid) mx = fmaxf(mx, __uint_as_float(r[i]));
        }
        const float m_cand = fmaxf(m_run, mx * c);
        bool resc = false;
        if (j == 0) {
          m_run = m_cand;
        } else if (m_cand > m_run) {
          alpha = ex2_approx(m_run - m_cand);
          m_run = m_cand;
          resc = true;
        }
        // O_t holds the sum over key blocks < j (P_t V_{j-1} completed before S_t of
        // block j was signalled), so it may be rescaled now.
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t r[32];
            tmem_load32(tO + cc * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_store32(tO + cc * 32, r);
          }
        }
        float unused = -INFINITY;
        if (kv_valid >= kBKV)
          softmax_row<false, false>(tS, kv_valid, c, -m_run, unused, psum, pk);
        else
          softmax_row<true, false>(tS, kv_valid, c, -m_run, unused, psum, pk);
      }
      l_run = l_run * alpha + psum;
      // P_t over S_t columns [0, 64): keys [2c, 2c + 1] in column c
      tmem_store32(tS, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
      tmem_store32(tS + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
      tmem_store_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[tile]);
    }
    if (ok) {
      // Output: O_t / l, rounded to bf16, staged in Q_t's shared memory (free once the last
      // QK is done, which precedes the last PV) in the 128-byte-swizzled layout Q was loaded
      // in, then written by two TMA stores (one per 64-column half; rows past n clipped).
      bool ok2 = mbar_wait_sleep(&o_done[tile], 0, wc, kSiteODone);
      ok2 = __all_sync(0xffffffffu, ok2);
      if (ok2) {
        tc_fence_after();
        const float inv_l = 1.0f / l_run;
        uint8_t* stage = smem + kOffQ + tile * kTileBytes;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t r[32];
          tmem_load32(tO + cc * 32, r);
          uint8_t* rowp = stage + (cc >> 1) * kHalfBytes + row * 128;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int chunk = (cc & 1) * 4 + i;  // 16-byte chunk of the 128-byte half-row
            *reinterpret_cast<uint4*>(rowp + ((chunk ^ (row & 7)) << 4)) =
                make_uint4(pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l),
                           pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l),
                           pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l),
                           pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l));
          }
        }
        fence_proxy_async_smem();  // the staged rows are visible to the TMA unit
        __syncwarp();
        if (lane == 0) mbar_arrive(&osync[tile]);
        bool ok3 = mbar_wait(&osync[tile], 0, wc, kSiteOSync);
        ok3 = __all_sync(0xffffffffu, ok3);
        if (ok3 && qq == 2 && lane == 0) {  // the tile's first warp (2 or 6)
          for (int h = 0; h < 2; ++h)
            tma_store_3d(&P.o_map, stage + h * kHalfBytes, head * 128 + h * 64, q0 + tile * kBQ, b);
          tma_store_commit_and_drain();
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// the shared-memory attribute has been raised on device d (set from any host thread)
std::atomic<bool> g_attr_set[16];

}  // namespace

cudaError_t launch_attention(int batch, int heads, int n, const bf16* q, const bf16* k, const bf16* v, bf16* out,
                             int ld_out, DeviceStatus* status, cudaStream_t s) {
  if (batch <= 0 || heads <= 0 || n <= 0) return cudaSuccess;
  AttnParams P;
  memset(&P, 0, sizeof(P));
  const uint64_t dims[3] = {128, (uint64_t)n, (uint64_t)batch * heads};
  const uint64_t str[2] = {256, (uint64_t)n * 256};
  const uint32_t box[3] = {64, 128, 1};
  if (!encode_tmap_bf16(&P.q_map, q, 3, dims, str, box)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&P.k_map, k, 3, dims, str, box)) return cudaErrorInvalidValue;
  if (!encode_tmap_bf16(&P.v_map, v, 3, dims, str, box)) return cudaErrorInvalidValue;
  const uint64_t odims[3] = {(uint64_t)ld_out, (uint64_t)n, (uint64_t)batch};
  const uint64_t ostr[2] = {(uint64_t)ld_out * 2, (uint64_t)n * ld_out * 2};
  if (!encode_tmap_bf16(&P.o_map, out, 3, odims, ostr, box)) return cudaErrorInvalidValue;
  P.out = out;
  P.ld_out = ld_out;
  P.n = n;
  P.heads = heads;
  P.scale_log2 = (float)(1.4426950408889634 / sqrt(128.0));
  P.status = status;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 16 && !g_attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e =
        cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    g_attr_set[dev].store(true, std::memory_order_release);
  }
  dim3 grid((n + 2 * kBQ - 1) / (2 * kBQ), heads, batch);
  LaunchScope scope(kClsAttention, s);
  return launch_k(attention_kernel, grid, dim3(kThreads), kSmemBytes, s, P);
}

}  // namespace dit
