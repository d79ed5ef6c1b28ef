// Small-token forward of a list of QLoRA linears in ONE launch (decode):
//   Y_p = X_p deq(W_p)^T + s_p (X_p A_p^T) B_p^T,   1 <= m_p <= 16 tokens,  1 <= r_p <= 128
//
// Glossary "QLoRA", "How QLoRA works": the frozen layer dequantises NF4 to bf16
// and adds the LoRA output; Day 25 notes, section 4.4: inference runs the
// 4-bit base with the adapter attached.  With a handful of tokens the step is a
// stream over the weight codes, so the kernel is built around keeping HBM busy
// and the chain of dependent steps inside one call short: a decoder layer
// makes four dependent calls (q,k,v | o | gate,up | down), each only a few
// microseconds of HBM time.
//
// Across calls (programmatic dependent launch): before it waits for the
// preceding kernel of the stream (griddepcontrol.wait), each CTA issues L2
// prefetches for the first tiles of its run and starts its cp.async ring on
// their code bytes -- weights, scales and B do not depend on the previous
// kernel.  So the codes are read before the wait: a kernel that writes a
// weight record must not let its dependents launch early (the quantiser's
// last kernel does not).  Right after the wait it lets the next kernel launch.
//
// Work: a TILE is 16 rows of one problem over the whole of k.  Tiles are
// dealt to the CTAs (two per SM) in contiguous runs of balanced cost; within a
// tile the 8 warps split the 64-wide absmax blocks of k into 8 contiguous
// ranges, and at the end of the tile their float32 partial sums are added in
// warp order in shared memory.  No tile is split between CTAs, so there is no
// cross-CTA reduction of Y and the result does not depend on the grid.
//
// X A^T is cut into at most 16 k-slices per problem (slice i on CTA i % grid,
// computed before the CTA's tiles); each slice's partial is published with a
// counter, and the first tile of a problem in a CTA's run waits (bounded) for
// them and adds them in slice order into sT = bf16(s X A^T), kept in shared
// memory for the following tiles of the problem.  The tile's epilogue then adds
// sT B^T (a float32 FMA chain in j order) and writes y.  Every CTA of the grid
// is resident at once (grid <= resident CTAs per SM x SMs), so the waits always end.
//
// A block of a warp: lanes stage the 16 rows x 32 code bytes into a per-warp
// shared-memory ring with cp.async (kDcRing - 2 blocks ahead, across tiles;
// the block's raw scale bytes ride the same ring);
// lane (g, q) then reads bytes 8q .. 8q+7 of rows g and g + 8 (elements 16q ..
// 16q+15 of the block) and turns each byte into its bf16 level pair with one
// lookup in a byte-indexed table, giving mma.sync m16n8k16 A fragments for the
// k permutation "MMA c, slots (2q, 2q+1) <- elements 16q+4c, +1; slots (2q+8,
// 2q+9) <- elements 16q+4c+2, +3"; the X fragment of the same permutation is
// X[tok][16q .. 16q+15], two 16-byte loads.  The block's product (8 tokens per
// MMA, 1 or 2 groups) is scaled by the block's restored scale a' in float32
// and added to the warp's sum.  So the effective weight is bf16(L[code]) * a'
// (within 2^-8 relative of the bf16_rn(L a') the fwd/bwd GEMMs use).
//
// Counters (per problem: X A^T slices published, tiles finished) are plain
// words updated with one atomic add each; the last finisher of a problem
// returns both to zero, so a workspace that starts zeroed stays zeroed across
// calls and graph replays.
#include <algorithm>
#include <cstdio>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kDcWarps = 8;
constexpr int kDcCtasPerSm = 2;            // two CTAs (16 warps) per SM hide the decode's latency
constexpr int kDcThreads = kDcWarps * 32;
constexpr int kDcTileRows = 16;            // rows per tile (the MMA's m)
constexpr int kDcRing = 12;                // cp.async ring depth per warp, in blocks (staged kDcRing - 2 ahead)
constexpr int kDcSlot = kDcTileRows * 32;  // one staged block: 16 rows x 32 code bytes, rows packed
constexpr int kDcScaleSlot = kDcTileRows * 4;  // and the aligned 4-byte word holding each row's raw scale
constexpr int kDcMaxProbs = 128;
constexpr int kDcMaxSlices = 16;           // X A^T slices per problem (each first tile adds them all)
constexpr int kDcPrefetchTiles = 4;        // tiles of its run a CTA keeps prefetched into L2 ahead
constexpr int kDcMaxCtas = 320;            // run table size (>= kDcCtasPerSm x SMs)
constexpr int kDcMaxR = 128;
// dynamic shared memory: code ring | scale ring | Y partials [2][warps][16 tok][16 rows] | sT [16 tok][128] (float)
constexpr size_t kDcCodeRingBytes = static_cast<size_t>(kDcWarps) * kDcRing * kDcSlot;
constexpr size_t kDcRingBytes = kDcCodeRingBytes + static_cast<size_t>(kDcWarps) * kDcRing * kDcScaleSlot;
constexpr size_t kDcRedBytes = 2ull * kDcWarps * 16 * 16 * 4;
constexpr size_t kDcTBytes = 16ull * kDcMaxR * 4;
constexpr size_t kDcDynSmem = kDcRingBytes + kDcRedBytes + kDcTBytes;

struct DcProb {
  const uint8_t* codes;
  const int8_t* absq;
  const float* step;
  const float* mean;
  const __nv_bfloat16* x;   // [m, k]
  const __nv_bfloat16* a;   // [r, k]
  const __nv_bfloat16* b;   // [n, r]
  __nv_bfloat16* y;         // [m, n]
  float* t_save;            // [m, r] or null
  float* tpart;             // [t_slices][16][r] partial X A^T
  unsigned* cnt;            // [2]: X A^T slices published, tiles finished (zero between calls)
  int n, k, m, r;
  float scale;
  int t_slices, t_w, s0;    // X A^T: slices of t_w 64-wide blocks, first global slice
  int tiles, u0;            // 16-row tiles, first global tile
};

struct DcParams {
  int count;
  int grid;
  int slices;                 // X A^T slices of the call
  unsigned long long wait_ns;
  unsigned* status;
  int run0[kDcMaxCtas + 1];   // CTA c takes the global tiles [run0[c], run0[c + 1])
  short sl0[kDcMaxCtas + 1];  // and computes the X A^T slices [sl0[c], sl0[c + 1]) first
  DcProb prob[kDcMaxProbs];
};

// (not volatile: a pure function of its operands, so the compiler may interleave independent MMAs)
__device__ __forceinline__ void dc_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
// A 16-byte load predicated in the instruction itself (zero when `on` is false; no branch).
__device__ __forceinline__ uint4 ldg_nc_v4_if(const void* p, bool on) {
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %4, 0;\n\t@q ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%5];\n\t}"
      : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
      : "r"(static_cast<int>(on)), "l"(p));
  return v;
}

// 4-byte cp.async issued only when `on` (predicated in the instruction; src-size 0 zero-fills)
__device__ __forceinline__ void cp_async4_if(uint32_t dst, const void* src, bool valid, bool on) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %3, 0;\n\t@q cp.async.ca.shared.global [%0], [%1], 4, %2;\n\t}" ::"r"(dst),
      "l"(src), "r"(valid ? 4 : 0), "r"(static_cast<int>(on))
      : "memory");
}

__device__ __forceinline__ void prefetch_l2_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// L2 prefetch of [p, p + bytes) by `nthr` threads (this one is `tid`): one plain prefetch per
// 128-byte line.
__device__ __forceinline__ void dc_prefetch_range(const void* p, int64_t bytes, int tid, int nthr) {
  if (bytes <= 0) return;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(127);
  const uintptr_t a1 = reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(bytes);
  for (uintptr_t a = a0 + static_cast<uintptr_t>(tid) * 128; a < a1; a += static_cast<uintptr_t>(nthr) * 128)
    prefetch_l2_line(reinterpret_cast<const void*>(a));
}

// Arrive on a counter (one atomic, no retry loop: many CTAs arrive on the same word); returns
// the count after this arrival.
__device__ __forceinline__ uint32_t dc_arrive(unsigned* c, unsigned v = 1u) { return atomicAdd(c, v) + v; }

__device__ __forceinline__ int dc_find_tile(const DcParams& p, int t) {  // problem of global tile t
  int lo = 0, hi = p.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.prob[mid].u0 <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}
__device__ __forceinline__ int dc_find_slice(const DcParams& p, int sl) {  // problem of X A^T slice sl
  int lo = 0, hi = p.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.prob[mid].s0 <= sl) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// First 64-wide block of warp w's share of a row of nbk blocks (the 8 warps take contiguous ranges).
__device__ __forceinline__ int dc_warp_block(int w, int nbk) { return (w * nbk) >> 3; }

// L2 prefetch of tile t_local of problem pr (codes, raw scales, rows of B) by the CTA's threads.
__device__ __forceinline__ void dc_prefetch_tile(const DcProb& pr, int t_local) {
  const int r0 = t_local * kDcTileRows, rows = min(kDcTileRows, pr.n - r0), nbk = pr.k >> 6;
  dc_prefetch_range(pr.codes + static_cast<int64_t>(r0) * (pr.k >> 1), static_cast<int64_t>(rows) * (pr.k >> 1),
                    threadIdx.x, kDcThreads);
  dc_prefetch_range(pr.absq + static_cast<int64_t>(r0) * nbk, static_cast<int64_t>(rows) * nbk, threadIdx.x,
                    kDcThreads);
  dc_prefetch_range(pr.b + static_cast<int64_t>(r0) * pr.r, static_cast<int64_t>(rows) * pr.r * 2, threadIdx.x,
                    kDcThreads);
  if (threadIdx.x == 0) {
    const int64_t s0 = (static_cast<int64_t>(r0) * nbk) >> 8, s1 = (static_cast<int64_t>(r0 + rows) * nbk - 1) >> 8;
    dc_prefetch_range(pr.step + s0, (s1 - s0 + 1) * 4, 0, 1);
  }
}

template <int NG>
__global__ void __launch_bounds__(kDcThreads, kDcCtasPerSm) k_decode(const __grid_constant__ DcParams p) {
  // level pairs of a code byte: s_lut[b * 32 + lane] = bf16 L[b >> 4] | (bf16 L[b & 15]) << 16, the
  // byte's two weights in mma fragment order; one column per lane, so lookups never conflict.  A
  // static array: a lookup is one shared load at [index + the table's fixed address].
  __shared__ __align__(16) uint32_t s_lut[256 * 32];
  __shared__ uint32_t s_lv[16];
  __shared__ int s_flag;
  extern __shared__ __align__(16) uint8_t s_dyn[];
  float* s_red = reinterpret_cast<float*>(s_dyn + kDcRingBytes);                 // [2][warps][16][16]
  float* s_t = reinterpret_cast<float*>(s_dyn + kDcRingBytes + kDcRedBytes);     // [16][kDcMaxR]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int t_begin = p.run0[blockIdx.x], t_end = p.run0[blockIdx.x + 1];

  // ---------------------------------------------------------------- prologue (before the wait)
  if (t_begin < t_end) {
    int pi = dc_find_tile(p, t_begin);
    for (int t = t_begin; t < t_end && t < t_begin + kDcPrefetchTiles; ++t) {
      if (t - p.prob[pi].u0 == p.prob[pi].tiles) ++pi;
      dc_prefetch_tile(p.prob[pi], t - p.prob[pi].u0);
    }
  }
  for (int sl = p.sl0[blockIdx.x]; sl < p.sl0[blockIdx.x + 1]; ++sl) {
    const DcProb& pr = p.prob[dc_find_slice(p, sl)];
    const int kb0 = (sl - pr.s0) * pr.t_w, kb1 = min(pr.k / 64, kb0 + pr.t_w);
    for (int j = warp; j < pr.r; j += kDcWarps)
      dc_prefetch_range(pr.a + static_cast<int64_t>(j) * pr.k + kb0 * 64, (kb1 - kb0) * 128, lane, 32);
  }
  {
    // the 16 bf16 levels go through shared memory (a dynamically indexed local array would put
    // the whole kernel on a stack frame)
    if (threadIdx.x < 16) {
      constexpr uint32_t hex[16] = QLORA_NF4_LEVELS_HEX;
      uint32_t v = 0;
#pragma unroll
      for (int c = 0; c < 16; ++c) v = threadIdx.x == c ? hex[c] : v;
      s_lv[threadIdx.x] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v)));
    }
    __syncthreads();
    // row b of the table is 32 copies of one word: 16-byte stores, 8 per thread
    for (int i = threadIdx.x; i < 256 * 8; i += kDcThreads) {
      const int b = i >> 3;
      const uint32_t v = s_lv[b >> 4] | (s_lv[b & 15] << 16);
      reinterpret_cast<uint4*>(s_lut)[i] = make_uint4(v, v, v, v);
    }
  }

  // ---- the cp.async stager: runs kDcRing - 2 blocks ahead of the consumer through the whole run
  // (tiles, then problems).  Per block, lane l copies bytes 16 (l & 1) .. +15 of row l >> 1, and
  // lane l < 16 the aligned 4-byte word of the raw scales that holds row l's scale of the block
  // (n % 8 == 0 makes the scale array a multiple of 8 bytes, so the word is inside it).
  const uint32_t ring0 = smem_u32(s_dyn) + warp * (kDcRing * kDcSlot);
  const uint32_t sring0 = smem_u32(s_dyn) + static_cast<uint32_t>(kDcCodeRingBytes) + warp * (kDcRing * kDcScaleSlot);
  const uint32_t stage_lane = ring0 + (lane >> 1) * 32 + (lane & 1) * 16;
  const uint32_t sstage_lane = sring0 + (lane & 15) * 4;
  int st_t = t_begin, st_pi = t_begin < t_end ? dc_find_tile(p, t_begin) : 0;
  int st_cnt = 0;        // ring slots left in the stager's current tile (its blocks rounded up to a pair)
  int st_real = 0;       // of which real blocks
  uint32_t st_off = 0;   // code ring slot offset (the scale slot is at st_off / 8)
  const uint8_t* st_src = nullptr;
  const int8_t* st_absq = nullptr;
  int64_t st_qf = 0;     // flattened scale index of row (lane & 15), current block
  bool st_ok = false, st_qok = false;
  // place the stager on the first tile at or after st_t where this warp has blocks
  auto st_enter = [&]() {
    st_cnt = 0;
    for (; st_t < t_end; ++st_t) {
      if (st_t - p.prob[st_pi].u0 == p.prob[st_pi].tiles) ++st_pi;
      const DcProb& pr = p.prob[st_pi];
      const int nbk = pr.k >> 6;
      const int kb = dc_warp_block(warp, nbk);
      st_real = dc_warp_block(warp + 1, nbk) - kb;
      if (st_real == 0) continue;
      st_cnt = (st_real + 1) & ~1;
      const int row0 = (st_t - pr.u0) * kDcTileRows;
      const int row = row0 + (lane >> 1);
      st_ok = row < pr.n;
      st_src = pr.codes + (st_ok ? static_cast<int64_t>(row) * (pr.k >> 1) + kb * 32 + (lane & 1) * 16 : 0);
      const int qrow = row0 + (lane & 15);
      st_qok = qrow < pr.n;
      st_absq = pr.absq;
      st_qf = st_qok ? static_cast<int64_t>(qrow) * nbk + kb : 0;
      return;
    }
  };
  // one ring slot: the next block's codes and scales (nothing in the pad slot of an odd range)
  auto stage_next = [&]() {
    if (st_cnt > 0) {
      if (st_real > 0) {
        cp_async16(stage_lane + st_off, st_src, st_ok);
        cp_async4_if(sstage_lane + (st_off >> 3), st_absq + (st_qf & ~int64_t(3)), st_qok, lane < 16);
        st_src += 32;
        ++st_qf;
        --st_real;
      }
      if (--st_cnt == 0) {
        ++st_t;
        st_enter();
      }
    }
    cp_async_commit();
    st_off = st_off + kDcSlot == kDcRing * kDcSlot ? 0u : st_off + kDcSlot;
  };
  st_enter();
  // kDcRing - 2 slots ahead: a pair is staged while the pair before it is still being read
  for (int i = 0; i < kDcRing - 2; ++i) stage_next();

  // X, the counters and the workspace may come from earlier kernels of the stream
  griddep_wait();
  griddep_launch_dependents();

  // ---------------------------------------------------------------- X A^T slices
  // slice sl (problem p, 64-wide blocks [kb0, kb1)): the 8 warps split its 16-k chunks, the CTA
  // adds their partial sums in warp order into the slice's partial
  for (int sl = p.sl0[blockIdx.x]; sl < p.sl0[blockIdx.x + 1]; ++sl) {
    const DcProb& pr = p.prob[dc_find_slice(p, sl)];
    const int si = sl - pr.s0;
    const int kb0 = si * pr.t_w, kb1 = min(pr.k / 64, kb0 + pr.t_w);
    const int nch = (kb1 - kb0) * 4;
    float* red = s_red;  // [warps][16 tok][16 j]
    for (int jg = 0; jg * 16 < pr.r; ++jg) {
      float acc[NG][4];
#pragma unroll
      for (int t = 0; t < NG; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
      const int j0 = jg * 16 + g, j1 = j0 + 8;
      for (int ch = warp; ch < nch; ch += kDcWarps) {
        const int kq = kb0 * 64 + ch * 16 + 4 * q;
        const uint2 a0 = j0 < pr.r ? ldg_nc_v2(pr.a + static_cast<int64_t>(j0) * pr.k + kq) : make_uint2(0u, 0u);
        const uint2 a1 = j1 < pr.r ? ldg_nc_v2(pr.a + static_cast<int64_t>(j1) * pr.k + kq) : make_uint2(0u, 0u);
#pragma unroll
        for (int t = 0; t < NG; ++t) {
          const int tok = t * 8 + g;
          const uint2 xb = tok < pr.m ? ldg_nc_v2(pr.x + static_cast<int64_t>(tok) * pr.k + kq) : make_uint2(0u, 0u);
          dc_mma(acc[t], a0.x, a1.x, a0.y, a1.y, xb.x, xb.y);
        }
      }
      // C fragment: d[0] = (row j0, tok 2q), d[1] = (j0, 2q+1), d[2] = (j1, 2q), d[3] = (j1, 2q+1)
#pragma unroll
      for (int t = 0; t < NG; ++t) {
        const int tk = t * 8 + 2 * q;
        red[(warp * 16 + tk) * 16 + g] = acc[t][0];
        red[(warp * 16 + tk + 1) * 16 + g] = acc[t][1];
        red[(warp * 16 + tk) * 16 + g + 8] = acc[t][2];
        red[(warp * 16 + tk + 1) * 16 + g + 8] = acc[t][3];
      }
      __syncthreads();
      {
        const int tok = threadIdx.x >> 4, j = threadIdx.x & 15;  // 256 threads = 16 tokens x 16 j
        if (tok < NG * 8 && jg * 16 + j < pr.r) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kDcWarps; ++w) v += red[(w * 16 + tok) * 16 + j];
          pr.tpart[(static_cast<int64_t>(si) * 16 + tok) * pr.r + jg * 16 + j] = v;
        }
      }
      __syncthreads();
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) dc_arrive(pr.cnt);  // count == t_slices: every slice partial of the problem is written
  }
  __syncthreads();  // s_lut written (a CTA without a slice gets here straight from the table fill)
  if (t_begin >= t_end) {
    cp_async_wait<0>();
    return;
  }

  // ---------------------------------------------------------------- tiles
  // one table lookup: the level pair of byte `i` of code word w (byte extracted with a permute,
  // then one multiply-add gives this lane's table address)
  const uint32_t lut_lane = smem_u32(s_lut) + static_cast<uint32_t>(lane) * 4u;
  auto lut = [&](uint32_t w, int i) -> uint32_t {
    const uint32_t b = __byte_perm(w, 0u, 0x4440u + i);
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(b * 128u + lut_lane));
    return v;
  };
  const unsigned char* ring_read = s_dyn + warp * (kDcRing * kDcSlot) + g * 32 + q * 8;
  const unsigned char* sring_read = s_dyn + kDcCodeRingBytes + warp * (kDcRing * kDcScaleSlot) + g * 4;
  uint32_t use_off = 0;  // ring slot offset of the consumer
  int cpi = dc_find_tile(p, t_begin);      // problem of the current tile
  int t_pi = -1;                           // problem whose sT is in s_t
  int pf_t = t_begin + kDcPrefetchTiles;   // next tile to prefetch into L2
  int pf_pi = cpi;
  int done_here = 0;                       // tiles of problem cpi finished by this CTA
  int buf = 0;
  bool alive = true;

  // the tiles-finished count of problem pi: the last finisher returns both counters to zero
  auto finish_problem = [&](int pi, int n_done) {
    if (threadIdx.x == 0 && n_done > 0) {
      const DcProb& pr = p.prob[pi];
      if (dc_arrive(pr.cnt + 1, static_cast<unsigned>(n_done)) == static_cast<uint32_t>(pr.tiles)) {
        *reinterpret_cast<volatile unsigned*>(pr.cnt) = 0u;
        *reinterpret_cast<volatile unsigned*>(pr.cnt + 1) = 0u;
      }
    }
  };

  for (int t = t_begin; t < t_end; ++t) {
    if (t - p.prob[cpi].u0 == p.prob[cpi].tiles) {
      finish_problem(cpi, done_here);
      done_here = 0;
      ++cpi;
    }
    const DcProb& pr = p.prob[cpi];
    const int row0 = (t - pr.u0) * kDcTileRows;
    const int nbk = pr.k >> 6;
    const int kb0 = dc_warp_block(warp, nbk), nb = dc_warp_block(warp + 1, nbk) - kb0;
    // rows g and g + 8 of the tile (past n: the stager zero-filled their codes and scales, and
    // their sums are never stored)
    const int ra = row0 + g < pr.n ? row0 + g : 0, rb = row0 + g + 8 < pr.n ? row0 + g + 8 : 0;
    const float mu = __ldg(pr.mean);
    // flattened block index f = row * nbk + kb: the raw scale is byte f & 3 of the staged word
    const int64_t fa = static_cast<int64_t>(ra) * nbk + kb0, fb = static_cast<int64_t>(rb) * nbk + kb0;
    const int fa3 = static_cast<int>(fa & 3), fb3 = static_cast<int>(fb & 3);
    // the float32 step of a block changes every 256 flattened blocks; a warp's range (< 256 blocks
    // for k <= 131072) meets at most one change: the two values and the j where it happens
    const int64_t nstep = (static_cast<int64_t>(pr.n) * nbk + 255) >> 8;
    const float sa0 = __ldg(pr.step + (fa >> 8)), sb0 = __ldg(pr.step + (fb >> 8));
    const float sa1 = (fa >> 8) + 1 < nstep ? __ldg(pr.step + (fa >> 8) + 1) : sa0;
    const float sb1 = (fb >> 8) + 1 < nstep ? __ldg(pr.step + (fb >> 8) + 1) : sb0;
    const int swa = static_cast<int>(256 - (fa & 255)), swb = static_cast<int>(256 - (fb & 255));
    // this lane's X rows: tokens tg * 8 + g (an absent token reads token 0: its column of the
    // product is never stored), elements 16 q .. 16 q + 15 of each block
    const uint4* xq[NG];
#pragma unroll
    for (int tg = 0; tg < NG; ++tg)
      xq[tg] = reinterpret_cast<const uint4*>(pr.x + static_cast<int64_t>(tg * 8 + g < pr.m ? tg * 8 + g : 0) * pr.k +
                                              16 * q + kb0 * 64);
    // this thread's row of B for the tile's epilogue (tokens tok < m, row row0 + rl), loaded now so
    // the epilogue does not wait for it; r <= 16 with 16-byte rows (otherwise read there)
    const int e_tok = threadIdx.x >> 4, e_row = row0 + (threadIdx.x & 15);
    const bool b_pre = (pr.r & 7) == 0 && pr.r <= 16 && e_tok < pr.m && e_row < pr.n;
    uint4 bpre[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
    if (b_pre) {
      const uint4* bq = reinterpret_cast<const uint4*>(pr.b + static_cast<int64_t>(e_row) * pr.r);
      bpre[0] = __ldg(bq);
      if (pr.r > 8) bpre[1] = __ldg(bq + 1);
    }
    float acc[NG][4];
#pragma unroll
    for (int tg = 0; tg < NG; ++tg) acc[tg][0] = acc[tg][1] = acc[tg][2] = acc[tg][3] = 0.f;
    // one block: j = its index in the warp's range, slot its code ring offset, u = 0 / 1 its place in the pair
    auto one_block = [&](int j, uint32_t slot, int u) {
      uint4 xv[NG][2];
#pragma unroll
      for (int tg = 0; tg < NG; ++tg) {
        xv[tg][0] = __ldg(xq[tg] + 8 * u);
        xv[tg][1] = __ldg(xq[tg] + 8 * u + 1);
      }
      // rows g and g + 8, bytes 8q .. 8q+7, and their scale words (plain shared loads: ordered
      // after the ring wait)
      const uint2 ca = *reinterpret_cast<const uint2*>(ring_read + slot);
      const uint2 cb = *reinterpret_cast<const uint2*>(ring_read + slot + 8 * 32);
      const uint32_t qwa = *reinterpret_cast<const uint32_t*>(sring_read + (slot >> 3));
      const uint32_t qwb = *reinterpret_cast<const uint32_t*>(sring_read + (slot >> 3) + 8 * 4);
      float blk[NG][4];
#pragma unroll
      for (int tg = 0; tg < NG; ++tg) blk[tg][0] = blk[tg][1] = blk[tg][2] = blk[tg][3] = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {  // h = 0: bytes 0..3 (MMAs 0, 1); h = 1: bytes 4..7 (MMAs 2, 3)
        const uint32_t wa = h ? ca.y : ca.x, wb = h ? cb.y : cb.x;
        const uint32_t a00 = lut(wa, 0), a01 = lut(wa, 1), a02 = lut(wa, 2), a03 = lut(wa, 3);
        const uint32_t b00 = lut(wb, 0), b01 = lut(wb, 1), b02 = lut(wb, 2), b03 = lut(wb, 3);
#pragma unroll
        for (int tg = 0; tg < NG; ++tg) {
          const uint4 x = xv[tg][h];
          dc_mma(blk[tg], a00, b00, a01, b01, x.x, x.y);
          dc_mma(blk[tg], a02, b02, a03, b03, x.z, x.w);
        }
      }
      const int sha = ((fa3 + j) & 3) * 8, shb = ((fb3 + j) & 3) * 8;
      const int qa = static_cast<int>(qwa << (24 - sha)) >> 24, qb = static_cast<int>(qwb << (24 - shb)) >> 24;
      const float aa = restore_absmax(static_cast<int8_t>(qa), j < swa ? sa0 : sa1, mu);
      const float ab = restore_absmax(static_cast<int8_t>(qb), j < swb ? sb0 : sb1, mu);
#pragma unroll
      for (int tg = 0; tg < NG; ++tg) {
        acc[tg][0] = fmaf(aa, blk[tg][0], acc[tg][0]);
        acc[tg][1] = fmaf(aa, blk[tg][1], acc[tg][1]);
        acc[tg][2] = fmaf(ab, blk[tg][2], acc[tg][2]);
        acc[tg][3] = fmaf(ab, blk[tg][3], acc[tg][3]);
      }
    };
    for (int j = 0; j < nb; j += 2) {
      stage_next();
      stage_next();
      cp_async_wait<kDcRing - 2>();  // this pair's two slots have landed
      __syncwarp();
      const uint32_t s0 = use_off, s1 = use_off + kDcSlot == kDcRing * kDcSlot ? 0u : use_off + kDcSlot;
      use_off = s1 + kDcSlot == kDcRing * kDcSlot ? 0u : s1 + kDcSlot;
      one_block(j, s0, 0);
      if (j + 1 < nb) one_block(j + 1, s1, 1);
      __syncwarp();  // the pair's slots are refilled by a later stage_next()
#pragma unroll
      for (int tg = 0; tg < NG; ++tg) xq[tg] += 16;
    }

    // ---- epilogue: the warps' partials in warp order, + sT B^T, -> y
    // C fragment: acc[tg][0] = (row g, tok 2q), [1] = (g, 2q+1), [2] = (g+8, 2q), [3] = (g+8, 2q+1)
    float* red = s_red + buf * (kDcWarps * 256);  // [warp][tok][row]
#pragma unroll
    for (int tg = 0; tg < NG; ++tg) {
      const int tk = tg * 8 + 2 * q;
      red[(warp * 16 + tk) * 16 + g] = acc[tg][0];
      red[(warp * 16 + tk + 1) * 16 + g] = acc[tg][1];
      red[(warp * 16 + tk) * 16 + g + 8] = acc[tg][2];
      red[(warp * 16 + tk + 1) * 16 + g + 8] = acc[tg][3];
    }
    if (cpi != t_pi) {
      // first tile of this problem in the run: wait for its X A^T slices, then sT into s_t
      if (threadIdx.x == 0) {
        const unsigned want = static_cast<unsigned>(pr.t_slices);
        bool ok = *reinterpret_cast<volatile unsigned*>(pr.cnt) >= want;
        if (!ok) {
          const uint64_t t0 = globaltimer_ns();
          for (uint32_t it = 1;; ++it) {
            if (*reinterpret_cast<volatile unsigned*>(pr.cnt) >= want) { ok = true; break; }
            if ((it & 63u) == 0 && globaltimer_ns() - t0 > p.wait_ns) break;
            __nanosleep(64);
          }
        }
        s_flag = ok;
        if (!ok) latch_status(p.status, ST_TIMEOUT);
      }
      __syncthreads();
      if (!s_flag) {
        alive = false;
        break;
      }
      __threadfence();
      const int64_t cstride = static_cast<int64_t>(16) * pr.r;
      for (int i = threadIdx.x; i < pr.m * pr.r; i += kDcThreads) {
        const int tok = i / pr.r, j = i - tok * pr.r;
        const float* src = pr.tpart + static_cast<int64_t>(tok) * pr.r + j;
        float xs[kDcMaxSlices];
#pragma unroll
        for (int c = 0; c < kDcMaxSlices; ++c) xs[c] = c < pr.t_slices ? __ldcg(src + c * cstride) : 0.f;
        float v = 0.f;
#pragma unroll
        for (int c = 0; c < kDcMaxSlices; ++c) v += xs[c];
        if (t == pr.u0 && pr.t_save) pr.t_save[i] = v;
        s_t[tok * kDcMaxR + j] = __bfloat162float(__float2bfloat16_rn(__fmul_rn(v, pr.scale)));
      }
      t_pi = cpi;
    }
    __syncthreads();
    {
      const int tok = threadIdx.x >> 4, rl = threadIdx.x & 15, row = row0 + rl;
      if (tok < pr.m && row < pr.n) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kDcWarps; ++w) v += red[(w * 16 + tok) * 16 + rl];
        const __nv_bfloat16* brow = pr.b + static_cast<int64_t>(row) * pr.r;
        const float* trow = s_t + tok * kDcMaxR;
        float l = 0.f;
        if (b_pre) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (h * 8 >= pr.r) break;
            const uint32_t w[4] = {bpre[h].x, bpre[h].y, bpre[h].z, bpre[h].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              l = fmaf(trow[h * 8 + 2 * e], __uint_as_float(w[e] << 16), l);
              l = fmaf(trow[h * 8 + 2 * e + 1], __uint_as_float(w[e] & 0xffff0000u), l);
            }
          }
        } else if ((pr.r & 7) == 0) {  // 16-byte rows: 8 values a load, the loads independent of the chain
#pragma unroll 4
          for (int j = 0; j < pr.r; j += 8) {
            const uint4 bv = __ldg(reinterpret_cast<const uint4*>(brow + j));
            const uint32_t w[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              l = fmaf(trow[j + 2 * e], __uint_as_float(w[e] << 16), l);
              l = fmaf(trow[j + 2 * e + 1], __uint_as_float(w[e] & 0xffff0000u), l);
            }
          }
        } else {
          for (int j = 0; j < pr.r; ++j) l = fmaf(trow[j], __bfloat162float(brow[j]), l);
        }
        pr.y[static_cast<int64_t>(tok) * pr.n + row] = __float2bfloat16_rn(v + l);
      }
    }
    buf ^= 1;
    ++done_here;
    // keep kDcPrefetchTiles tiles of the run prefetched into L2
    if (pf_t < t_end) {
      if (pf_t - p.prob[pf_pi].u0 >= p.prob[pf_pi].tiles) pf_pi = dc_find_tile(p, pf_t);
      dc_prefetch_tile(p.prob[pf_pi], pf_t - p.prob[pf_pi].u0);
      ++pf_t;
    }
  }
  cp_async_wait<0>();
  if (alive) finish_problem(cpi, done_here);
}

// ---------------------------------------------------------------------------- host
int decode_max_problems() { return kDcMaxProbs; }

namespace {
struct DcPlan {
  int grid, slices, tiles;
  size_t ws_bytes;
  std::vector<int> run0, sl0;
  std::vector<size_t> off_cnt, off_tpart;
  std::vector<int> t_slices, t_w, s0, ptiles, u0;
};

size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

// CTAs of the kernel resident per SM (the waits inside need the whole grid resident at once).
int dc_ctas_per_sm() {
  static int cached = -1;
  if (cached < 0) {
    int a = 0, b = 0;
    if (cudaFuncSetAttribute(k_decode<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kDcDynSmem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_decode<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kDcDynSmem)) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, k_decode<1>, kDcThreads, kDcDynSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_decode<2>, kDcThreads, kDcDynSmem) != cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
    const int c = a < b ? a : b;
    cached = c < 1 ? 1 : (c > kDcCtasPerSm ? kDcCtasPerSm : c);
  }
  return cached;
}

DcPlan dc_plan(const GroupedProblem* probs, int count, int num_sms) {
  DcPlan pl;
  const int sms = num_sms > 0 ? num_sms : 1;
  pl.t_slices.resize(count);
  pl.t_w.resize(count);
  pl.s0.resize(count);
  pl.ptiles.resize(count);
  pl.u0.resize(count);
  // 16-row tiles; a tile's cost is its 64-wide blocks plus a fixed share for its epilogue
  int t = 0;
  double cost = 0.0;
  std::vector<double> tile_cost(static_cast<size_t>(count));
  for (int i = 0; i < count; ++i) {
    pl.ptiles[i] = static_cast<int>((probs[i].w.n + kDcTileRows - 1) / kDcTileRows);
    pl.u0[i] = t;
    t += pl.ptiles[i];
    tile_cost[static_cast<size_t>(i)] = static_cast<double>(probs[i].w.k / 64) + 2.0;
    cost += tile_cost[static_cast<size_t>(i)] * pl.ptiles[i];
  }
  pl.tiles = t;
  int slots = sms * dc_ctas_per_sm();  // every CTA of the grid resident at once
  if (slots > kDcMaxCtas) slots = kDcMaxCtas;
  const int tile_ctas = t < slots ? t : slots;
  // contiguous runs of balanced cost over the tile CTAs: CTA c starts at the first tile whose cost
  // prefix reaches c / tile_ctas of the total
  std::vector<int> run0(static_cast<size_t>(tile_ctas) + 1, t);
  {
    int c = 0;
    double pre = 0.0;
    for (int i = 0; i < count && c < tile_ctas; ++i)
      for (int lt = 0; lt < pl.ptiles[i] && c < tile_ctas; ++lt) {
        while (c < tile_ctas && pre >= cost * c / tile_ctas) run0[static_cast<size_t>(c++)] = pl.u0[i] + lt;
        pre += tile_cost[static_cast<size_t>(i)];
      }
  }
  // X A^T slices: about one per tile CTA over the whole list, in proportion to each problem's r k
  double work = 0.0;
  for (int i = 0; i < count; ++i) work += static_cast<double>((probs[i].r + 15) / 16) * probs[i].w.k;
  int sl = 0;
  for (int i = 0; i < count; ++i) {
    const int blocks = static_cast<int>(probs[i].w.k / 64);
    const double share = static_cast<double>((probs[i].r + 15) / 16) * probs[i].w.k / work;
    int want = static_cast<int>(share * tile_ctas + 0.5);
    want = want < 1 ? 1 : (want > blocks ? blocks : want);
    if (want > kDcMaxSlices) want = kDcMaxSlices;
    pl.t_w[i] = (blocks + want - 1) / want;
    pl.t_slices[i] = (blocks + pl.t_w[i] - 1) / pl.t_w[i];
    pl.s0[i] = sl;
    sl += pl.t_slices[i];
  }
  pl.slices = sl;
  // Who computes the slices (they come first in a CTA, so they delay its tiles): CTAs of their own
  // when the grid has room for them, else the tile CTAs whose runs cost least, a contiguous range
  // of slices each.
  const int extra = t < slots ? std::min(slots - t, sl) : 0;
  pl.grid = tile_ctas + extra;
  pl.run0 = run0;
  pl.run0.resize(static_cast<size_t>(pl.grid) + 1, t);
  for (int c = tile_ctas; c <= pl.grid; ++c) pl.run0[static_cast<size_t>(c)] = t;
  std::vector<int> who;  // the slice CTAs
  if (extra > 0) {
    for (int c = tile_ctas; c < pl.grid; ++c) who.push_back(c);
  } else {
    // cost prefix over the tiles, then each run's cost in O(1)
    std::vector<double> cpre(static_cast<size_t>(t) + 1, 0.0);
    for (int i = 0, tt = 0; i < count; ++i)
      for (int lt = 0; lt < pl.ptiles[i]; ++lt, ++tt)
        cpre[static_cast<size_t>(tt) + 1] = cpre[static_cast<size_t>(tt)] + tile_cost[static_cast<size_t>(i)];
    std::vector<std::pair<double, int>> by_cost;
    by_cost.reserve(static_cast<size_t>(tile_ctas));
    for (int c = 0; c < tile_ctas; ++c)
      by_cost.push_back({cpre[static_cast<size_t>(run0[static_cast<size_t>(c) + 1])] -
                             cpre[static_cast<size_t>(run0[static_cast<size_t>(c)])],
                         c});
    std::stable_sort(by_cost.begin(), by_cost.end(),
                     [](const std::pair<double, int>& a, const std::pair<double, int>& b) { return a.first < b.first; });
    const int e = std::min(sl, tile_ctas);
    for (int k = 0; k < e; ++k) who.push_back(by_cost[static_cast<size_t>(k)].second);
    std::sort(who.begin(), who.end());
  }
  std::vector<int> nsl(static_cast<size_t>(pl.grid), 0);
  for (size_t k = 0; k < who.size(); ++k)
    nsl[static_cast<size_t>(who[k])] = static_cast<int>((static_cast<long long>(k + 1) * sl) / static_cast<long long>(who.size()) -
                                                        (static_cast<long long>(k) * sl) / static_cast<long long>(who.size()));
  pl.sl0.assign(static_cast<size_t>(pl.grid) + 1, 0);
  for (int c = 0; c < pl.grid; ++c) pl.sl0[static_cast<size_t>(c) + 1] = pl.sl0[static_cast<size_t>(c)] + nsl[static_cast<size_t>(c)];
  size_t off = 0;
  pl.off_cnt.resize(count);
  pl.off_tpart.resize(count);
  for (int i = 0; i < count; ++i) {
    pl.off_cnt[i] = off;
    off += al256(2 * 4);
    pl.off_tpart[i] = off;
    off += al256(static_cast<size_t>(pl.t_slices[i]) * 16 * probs[i].r * 4);
  }
  pl.ws_bytes = off;
  return pl;
}
}  // namespace

size_t decode_workspace_bytes(const GroupedProblem* probs, int count, int num_sms) {
  return dc_plan(probs, count, num_sms).ws_bytes;
}

cudaError_t launch_decode(const GroupedProblem* probs, int count, void* ws, unsigned* status, uint64_t wait_ns,
                          int num_sms, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  const DcPlan pl = dc_plan(probs, count, num_sms);
  static DcParams prm;  // 20+ KB: not on the host stack; launches copy it
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  prm.count = count;
  prm.grid = pl.grid;
  prm.slices = pl.slices;
  prm.wait_ns = wait_ns;
  prm.status = status;
  for (int c = 0; c <= pl.grid; ++c) {
    prm.run0[c] = pl.run0[static_cast<size_t>(c)];
    prm.sl0[c] = static_cast<short>(pl.sl0[static_cast<size_t>(c)]);
  }
  int mmax = 1;
  char* base = static_cast<char*>(ws);
  for (int i = 0; i < count; ++i) {
    const GroupedProblem& g = probs[i];
    DcProb& d = prm.prob[i];
    d.codes = g.w.codes;
    d.absq = g.w.absq;
    d.step = g.w.step;
    d.mean = g.w.mean;
    d.x = g.x;
    d.a = g.lora_a;
    d.b = g.lora_b;
    d.y = g.y;
    d.t_save = g.t_save;
    d.tpart = reinterpret_cast<float*>(base + pl.off_tpart[i]);
    d.cnt = reinterpret_cast<unsigned*>(base + pl.off_cnt[i]);
    d.n = static_cast<int>(g.w.n);
    d.k = static_cast<int>(g.w.k);
    d.m = g.m;
    d.r = g.r;
    d.scale = g.alpha / static_cast<float>(g.r);
    d.t_slices = pl.t_slices[i];
    d.t_w = pl.t_w[i];
    d.s0 = pl.s0[i];
    d.tiles = pl.ptiles[i];
    d.u0 = pl.u0[i];
    if (g.m > mmax) mmax = g.m;
  }
  cudaError_t e0 =
      mmax <= 8 ? set_smem_limit_once(k_decode<1>, kDcDynSmem) : set_smem_limit_once(k_decode<2>, kDcDynSmem);
  if (e0 != cudaSuccess) return e0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kDcThreads);
  cfg.dynamicSmemBytes = kDcDynSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = mmax <= 8 ? cudaLaunchKernelEx(&cfg, k_decode<1>, prm) : cudaLaunchKernelEx(&cfg, k_decode<2>, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace qlora
