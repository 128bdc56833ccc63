// Shared device helpers for the sm_103a kernels: mbarriers with bounded waits, TMA tile
// loads, tcgen05 (TMEM allocation, MMA, commit, TMEM loads/stores) and the shared-memory
// matrix / instruction descriptors of the 5th-generation tensor cores.  All inline PTX is
// written from the public PTX ISA description of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dit {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------------
// Device status word (first bytes of every workspace).  Kernels never trap: a wait
// that runs past its limit sets a bit here, the kernel unwinds, and the host reports
// DIT_ERR_TIMEOUT from dit_sync_status().
// ---------------------------------------------------------------------------------
enum : uint32_t { kStatusTimeout = 1u, kStatusBadLaunch = 2u };

struct DeviceStatus {
  uint32_t word;     // OR of kStatus* bits
  uint32_t where;    // id of the first wait that gave up (kernel * 16 + site)
  uint32_t pad[62];
};

// ---------------------------------------------------------------------------------
// Small utilities
// ---------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // RNE, lo in the low half
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

// ---------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait limits.  A wait that has not completed after kWaitLimitNs marks the status
// word, raises the block's abort flag and returns false; every role polls the abort
// flag so the whole block unwinds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

struct WaitCtx {
  DeviceStatus* status;
  volatile int* abort_flag;  // in shared memory
  uint64_t limit_ns;
};

static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*w.abort_flag) return false;
      if (global_timer_ns() - t0 > w.limit_ns) {
        if (w.status && atomicOr(&w.status->word, kStatusTimeout) == 0u) atomicExch(&w.status->where, site);
        *w.abort_flag = 1;
        __threadfence_block();
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  if (mbar_try(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, w, site);
}

// The same bounded wait for warps that have nothing else to do meanwhile: try_wait with a
// suspend-time hint lets the thread sleep in hardware until the phase completes (or the hint
// elapses) instead of spinning on issue slots that a computing or MMA-issuing warp of the
// same SM sub-partition needs.  The limit and abort checks run after every return.
constexpr uint32_t kSleepHintNs = 1000000u;  // 1 ms

__device__ __forceinline__ bool mbar_try_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSleepHintNs)
      : "memory");
  return ok != 0;
}

static __device__ __noinline__ bool mbar_wait_sleep_slow(uint64_t* bar, uint32_t parity, const WaitCtx& w,
                                                         uint32_t site) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_sleep(bar, parity)) return true;
    if (*w.abort_flag) return false;
    if (global_timer_ns() - t0 > w.limit_ns) {
      if (w.status && atomicOr(&w.status->word, kStatusTimeout) == 0u) atomicExch(&w.status->where, site);
      *w.abort_flag = 1;
      __threadfence_block();
      return false;
    }
  }
}

__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity, const WaitCtx& w, uint32_t site) {
  if (mbar_try_sleep(bar, parity)) return true;
  return mbar_wait_sleep_slow(bar, parity, w, site);
}

// ---------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) tile loads into shared memory, completing on an mbarrier.
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Generic-proxy writes to shared memory (st.shared) made visible to the async proxy
// (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------
// tcgen05: Tensor Memory and the 5th-generation MMA
// ---------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A/B and an fp32 accumulator.
// Bits: [4,6) D format (1 = f32), [7,10) A format (1 = bf16), [10,13) B format
// (1 = bf16), 15 A major (0 = K), 16 B major (0 = K, 1 = MN), [17,23) N >> 3,
// [24,29) M >> 4.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
// Bits: [0,14) start address >> 4, [16,30) leading byte offset >> 4, [32,46) stride
// byte offset >> 4, [46,49) = 0b001, [61,64) swizzle mode (2 = 128-byte).
// K-major: rows of 128 B (64 bf16 along K), 8-row groups SBO apart; LBO unused.
// MN-major: 128 B along M/N per K-row; LBO = distance between 64-element MN blocks,
// SBO = distance between 8-row K groups.
__device__ __forceinline__ uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// 32 TMEM lanes x 32 consecutive 32-bit columns: thread t of the warp receives lane
// (warp's lane quarter base + t), columns [col, col + 32).
#define DIT_R32(r)                                                                                             \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),   \
      "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),    \
      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),   \
      "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define DIT_RW32(r)                                                                                            \
  "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]),   \
      "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),    \
      "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),   \
      "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
#define DIT_IN32(r)                                                                                            \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), \
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),           \
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),           \
      "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

// Load then wait; the wait names the registers so that no use is scheduled before it.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : DIT_R32(r)
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" : DIT_RW32(r) : : "memory");
}

__device__ __forceinline__ void tmem_store32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      DIT_IN32(r)
      : "memory");
}

__device__ __forceinline__ void tmem_store_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x with the hardware approximation (MUFU.EX2), flushing subnormals to zero.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialisation
// may start while its predecessor on the stream still runs.  grid_dependency_wait() blocks
// until every prerequisite grid has completed and its memory is visible; nothing before it
// may read or write memory that an earlier kernel writes or reads.  allow_dependents()
// lets the next kernel on the stream start launching (it still waits in its own
// grid_dependency_wait()).  Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace dit
