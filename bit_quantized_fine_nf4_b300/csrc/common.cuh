// Device helpers shared by the sm_103a kernels of the NF4 QLoRA linear:
// status word, bounded mbarrier waits, TMA, tcgen05 (TMEM alloc / MMA / ld / st),
// shared-memory matrix descriptors and the NF4 block decode.
//
// Every wait on an mbarrier is bounded in time (globaltimer).  On expiry the
// kernel latches QLORA_ST_TIMEOUT in the status word, raises a per-CTA abort
// flag so the other roles stop waiting, frees its TMEM and returns.  Nothing
// here traps.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <set>
#include <utility>

#include "kernels.h"

namespace qlora {

// ------------------------------------------------------------------ status
// (bits ST_* are declared in kernels.h)
__device__ __forceinline__ void latch_status(unsigned* status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Wait until the phase with parity `parity` of `bar` has completed.  Returns
// false if `limit_ns` elapsed first or another role of the CTA aborted.
// Cluster-scope acquire: for phases completed by arrivals from the peer CTA.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

template <bool kClusterScope = false>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                          volatile int* abort_flag) {
  auto poll = [&]() { return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (poll()) return true;
    if ((it & 31u) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (globaltimer_ns() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// A bounded wait expired: latch the status and make the CTA's other roles stop waiting.
__device__ __forceinline__ void abort_cta(unsigned* status, int* abort_flag) {
  latch_status(status, ST_TIMEOUT);
  *reinterpret_cast<volatile int*>(abort_flag) = 1;
}

// ------------------------------------------------------------------ programmatic dependent launch
// Every kernel here keeps two rules, which together order a chain of such launches:
//  * it calls griddep_launch_dependents only after its own griddep_wait has returned, so when the
//    next kernel starts, every kernel before this one has completed;
//  * before its griddep_wait it reads nothing the immediately preceding kernel writes (only data
//    of earlier kernels, the frozen NF4 record, or its own parameters) and writes nothing.
// Let the next kernel in the stream start launching now (it still has to wait
// with griddep_wait before it reads anything this grid writes).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the grids this one depends on have completed and their writes are visible.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Host: a plain launch with programmatic stream serialization (the kernel must call griddep_wait
// before it touches memory the preceding kernels of the stream may still use).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_plain(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ------------------------------------------------------------------ proxies / fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tiled load of one box into shared memory, completing tx bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// ------------------------------------------------------------------ TMEM
// Whole warp: allocate `ncols` (power of two >= 32) TMEM columns; the base
// address is written to `dst` in shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive (once) on `bar` when every MMA issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// ------------------------------------------------------------------ CTA pairs (clusters of two)
// The two CTAs of a cluster of size 2 sit on the two SMs of one TPC; with
// cta_group::2 one thread of the even CTA issues MMAs with M = 256 whose A rows
// 0..127 / 128..255 and B columns [0, N/2) / [N/2, N) come from the shared
// memory of CTA 0 / CTA 1, and whose accumulator rows land in each CTA's own
// TMEM.  Every tcgen05 instruction of such a kernel uses cta_group::2.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// All threads of both CTAs.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive (release, cluster scope) on the barrier at the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* bar, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}
// One warp in each CTA of the pair, together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_pair_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the barrier at this offset in every CTA of `cta_mask` when all
// MMAs issued so far by this thread are done.
__device__ __forceinline__ void mma_pair_commit_multicast(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

#define QLORA_R8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), "r"(r[b + 4]), "r"(r[b + 5]), \
                    "r"(r[b + 6]), "r"(r[b + 7])
#define QLORA_W8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), "=r"(r[b + 4]), \
                    "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])

// Warp-collective: thread i reads TMEM lane (lane field of taddr) + i, 32 consecutive columns.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : QLORA_W8(0), QLORA_W8(8), QLORA_W8(16), QLORA_W8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : QLORA_W8(0), QLORA_W8(8)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Warp-collective: thread i writes TMEM lane (lane field of taddr) + i, 32 consecutive columns.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      QLORA_R8(0), QLORA_R8(8), QLORA_R8(16), QLORA_R8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor for tcgen05 with the 128-byte swizzle:
// start address, leading-dimension byte offset, stride-dimension byte offset
// (all >> 4), the fixed 0b001 field at bit 46, swizzle mode 2 (128 B) at bit 61.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo_bytes & 0x3FFFFu) >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, dense.
// a_mn / b_mn: operand is MN-major (1) or K-major (0).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a tile whose rows
// are 128 bytes, stored with the 128-byte swizzle (tile base 1024-aligned).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// ------------------------------------------------------------------ NF4
// The 16 NF4 levels as float32 bit patterns: quantiles of N(0,1) with an exact
// zero, normalised to [-1, 1] (Ultralytics glossary "QLoRA", "How QLoRA
// works"), evaluated in double precision and rounded once to float.
#define QLORA_NF4_L0 (-1.0f)
#define QLORA_NF4_LEVELS_HEX                                                                          \
  {0xbf800000u, 0xbf3239b3u, 0xbf066b30u, 0xbeca32a0u, 0xbe91a24cu, 0xbe3d353fu, 0xbdba786bu, 0x00000000u, \
   0x3da2fb03u, 0x3e24cae1u, 0x3e7c04dcu, 0x3ead0338u, 0x3ee1a4b7u, 0x3f1007aau, 0x3f3913b1u, 0x3f800000u}

__device__ __forceinline__ float nf4_level(int j) {
  constexpr uint32_t hex[16] = QLORA_NF4_LEVELS_HEX;
  return __uint_as_float(hex[j]);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Restored block scale a' = float(q) * step + mu (two separate float32 roundings).
__device__ __forceinline__ float restore_absmax(int8_t q, float step, float mu) {
  return __fadd_rn(__fmul_rn(static_cast<float>(q), step), mu);
}

// Byte planes of the 16-entry table V[j] = bf16_rn(L[j] * a'):
// lo[p] / hi[p] hold the low / high bytes of V[4p .. 4p+3].
struct Nf4Table {
  uint32_t lo[4], hi[4];
};

__device__ __forceinline__ Nf4Table nf4_table(float a2) {
  constexpr uint32_t hex[16] = QLORA_NF4_LEVELS_HEX;
  uint32_t p[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float v0 = __fmul_rn(__uint_as_float(hex[2 * j]), a2);
    const float v1 = __fmul_rn(__uint_as_float(hex[2 * j + 1]), a2);
    p[j] = pack_bf16x2_rn(v0, v1);  // V[2j] low half, V[2j+1] high half
  }
  Nf4Table t;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    t.lo[q] = prmt(p[2 * q], p[2 * q + 1], 0x6420u);
    t.hi[q] = prmt(p[2 * q], p[2 * q + 1], 0x7531u);
  }
  return t;
}

// Decode one 32-bit word of packed codes (8 elements; byte b holds element 2b
// in its high nibble and 2b+1 in its low nibble) into 4 bf16x2 words, element
// order preserved (element 2i in the low half of out[i]).
__device__ __forceinline__ void nf4_decode_word(const Nf4Table& t, uint32_t w, uint32_t (&out)[4]) {
  const uint32_t s7 = w & 0x77777777u;                       // level index within its half-table
  const uint32_t pick = ((w & 0x88888888u) >> 1) | 0x32103210u;  // byte i from lower (i) or upper (i+4)
  uint32_t sel = s7, ch = pick;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t lo_a = prmt(t.lo[0], t.lo[1], sel);
    const uint32_t lo_b = prmt(t.lo[2], t.lo[3], sel);
    const uint32_t hi_a = prmt(t.hi[0], t.hi[1], sel);
    const uint32_t hi_b = prmt(t.hi[2], t.hi[3], sel);
    const uint32_t lo = prmt(lo_a, lo_b, ch);  // bytes in nibble order: e1, e0, e3, e2
    const uint32_t hi = prmt(hi_a, hi_b, ch);
    out[2 * h + 0] = prmt(lo, hi, 0x4051u);    // (e0, e1)
    out[2 * h + 1] = prmt(lo, hi, 0x6273u);    // (e2, e3)
    sel = s7 >> 16;
    ch = pick >> 16;
  }
}

// Decode a whole 64-element block (32 code bytes) into 32 bf16x2 words.
__device__ __forceinline__ void nf4_decode_block(const uint4& c0, const uint4& c1, float a2, uint32_t (&out)[32]) {
  const Nf4Table t = nf4_table(a2);
  const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t o[4];
    nf4_decode_word(t, w[i], o);
    out[4 * i + 0] = o[0];
    out[4 * i + 1] = o[1];
    out[4 * i + 2] = o[2];
    out[4 * i + 3] = o[3];
  }
}

// 16-byte cp.async (L2 only); src-size 0 when !valid zero-fills the destination
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void sts_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// 64 LoRA B entries B[row, jb .. jb+63] as 32 bf16x2 words (zero past r or
// past the last row).  B is [n_rows, r] row-major: with r even its rows start
// on 4-byte boundaries and are read in 32-bit words; with r odd, element by element.
__device__ __forceinline__ void load_lora_b_row(const __nv_bfloat16* lora_b, int row, int n_rows, int r, int jb,
                                                uint32_t (&words)[32]) {
  const bool row_ok = row < n_rows;
  if ((r & 1) == 0) {
    const uint32_t* brow = reinterpret_cast<const uint32_t*>(lora_b + static_cast<int64_t>(row) * r);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int j = jb + 2 * c;
      words[c] = (row_ok && j < r) ? brow[j >> 1] : 0u;
    }
  } else {
    const unsigned short* b16 = reinterpret_cast<const unsigned short*>(lora_b) + static_cast<int64_t>(row) * r;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int j = jb + 2 * c;
      const uint32_t lo = (row_ok && j < r) ? b16[j] : 0u;
      const uint32_t hi = (row_ok && j + 1 < r) ? b16[j + 1] : 0u;
      words[c] = lo | (hi << 16);
    }
  }
}

// Host: raise a kernel's dynamic shared-memory limit once per (kernel, device)
// (the attribute call is host work; repeating it on every launch costs
// microseconds).  Keyed by the kernel's address: template instances of one
// kernel share a function type but not an address.
inline bool smem_limit_done(const void* kernel, int device, bool mark) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lk(mu);
  const auto key = std::make_pair(kernel, device);
  if (mark) {
    done.insert(key);
    return true;
  }
  return done.count(key) != 0;
}

template <typename Kernel>
inline cudaError_t set_smem_limit_once(Kernel* kernel, size_t bytes) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  const void* key = reinterpret_cast<const void*>(kernel);
  if (smem_limit_done(key, d, false)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) smem_limit_done(key, d, true);
  return e;
}

}  // namespace qlora
