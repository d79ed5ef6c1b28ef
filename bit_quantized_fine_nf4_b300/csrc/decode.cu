// Small-token forward of a list of QLoRA linears in ONE launch (decode):
//   Y_p = X_p deq(W_p)^T + s_p (X_p A_p^T) B_p^T,   1 <= m_p <= 16 tokens,  1 <= r_p <= 128
//
// Glossary "QLoRA", "How QLoRA works": the frozen layer dequantises NF4 to bf16
// and adds the LoRA output; Day 25 notes, section 4.4: inference runs the
// 4-bit base with the adapter attached.  With a handful of tokens the step is a
// stream over the weight codes, so the kernel is built around keeping HBM busy
// across calls: a decoder layer makes four dependent calls (q,k,v | o |
// gate,up | down), each only a few microseconds of HBM time.
//
// Across calls (programmatic dependent launch): each CTA first issues L2
// prefetches for every code byte it will read -- the weights do not depend on
// the previous kernel -- and only then waits (griddepcontrol.wait) for the
// preceding kernel of the stream; right after that wait it lets the next
// kernel launch, which prefetches its own weights while this one computes.
//
// Work: the list is cut into units of equal size -- T units (problem, a range
// of k) that compute partial X A^T, placed first, then W units (problem, tile
// of 128 rows, 256 k) -- and every CTA (one per SM) takes one contiguous run of
// units.  A run accumulates the units of one row tile in registers; a tile
// split between runs leaves float32 partials that the last arriving CTA adds in
// run order (deterministic).  The tile's finaliser adds the LoRA term with
// sT = bf16(s T), which the last T unit of the problem publishes; finalisers
// that get there first wait for it (bounded wait; every CTA of the grid is
// resident: the grid has at most one CTA per SM and the next kernel can only
// launch after every CTA of this one has started).
//
// A W unit: warp w owns rows 16w .. 16w+15 of the tile; per 64-wide absmax
// block, lanes stage the 16 rows x 32 code bytes into a shared-memory ring with
// cp.async (kDcRing blocks ahead), decode them with the byte-permute table of
// the bf16 NF4 levels into mma.sync m16n8k16 A fragments (k permuted so lane
// (g, q) holds k = 16c + 4q .. 4q+3 of chunk c), and multiply with the X
// fragments (8 tokens per MMA, 1 or 2 groups) into a per-block accumulator,
// which is scaled by the block's restored scale a' and added to the run's sum.
// So the effective weight is bf16(L[code]) * a' with a' applied in float32 to
// the block's partial sums (within 2^-8 relative of the bf16_rn(L a') the
// fwd/bwd GEMMs use).
//
// Counters are 64-bit (call epoch, count): a word left by another call (or
// never initialised) is reset by its first arriver, and every counter is
// returned to (epoch, 0) by its last user, so graph replays of one call work.
#include <algorithm>
#include <cstdio>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kDcWarps = 8;
constexpr int kDcThreads = kDcWarps * 32;
constexpr int kDcRows = kDcWarps * 16;     // rows per tile
constexpr int kDcUnitBlocks = 4;           // 64-wide blocks per W unit (256 k)
constexpr int kDcRing = 6;                 // cp.async ring depth per warp, in blocks
constexpr int kDcPitch = 48;               // shared-memory bytes per staged row piece (32 used, padded: no bank conflicts)
constexpr int kDcStage = 16 * kDcPitch;    // one block of the warp's 16 rows
constexpr int kDcMaxProbs = 128;
constexpr int kDcTChunk = 256;             // k per T sub-chunk

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
  float* tpart;             // [t_units][16][r] partial X A^T
  __nv_bfloat16* st;        // [16][r] bf16(s T)
  float* ypart;             // [tiles][maxseg][16][128] partial Y
  unsigned long long* cnt;  // [2 + tiles]: T, tiles done, then one per tile
  int n, k, m, r;
  float scale;
  int t_units, t_sub;       // T units and 256-k sub-chunks per T unit
  int tiles, ku;            // row tiles, W units per tile (k / 256)
  int u0_t, u0_w;           // first T unit, first W unit (global unit index)
};

struct DcParams {
  int count;
  int grid;
  int maxseg;
  uint32_t epoch;
  long long units;            // all units of the call
  unsigned long long wait_ns;
  unsigned* status;
  DcProb prob[kDcMaxProbs];
};

__device__ __forceinline__ void dc_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// First unit of CTA c when `units` units are dealt to `grid` CTAs in contiguous runs.
__device__ __forceinline__ long long dc_run_start(int c, long long units, int grid) {
  return static_cast<long long>(c) * units / grid;
}
// CTA whose run holds unit u.
__device__ __forceinline__ int dc_cta_of(long long u, long long units, int grid) {
  return static_cast<int>(((u + 1) * grid - 1) / units);
}

// Arrive on a (epoch, count) counter; returns the count after this arrival.
__device__ __forceinline__ uint32_t dc_arrive(unsigned long long* c, uint32_t epoch) {
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(c);
  for (;;) {
    const uint32_t cnt = static_cast<uint32_t>(old >> 32) == epoch ? static_cast<uint32_t>(old) : 0u;
    const unsigned long long want = (static_cast<unsigned long long>(epoch) << 32) | (cnt + 1u);
    const unsigned long long prev = atomicCAS(c, old, want);
    if (prev == old) return cnt + 1u;
    old = prev;
  }
}

__device__ __forceinline__ int dc_find_prob(const DcParams& p, long long u, bool t_unit) {
  int lo = 0, hi = p.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const long long s = t_unit ? p.prob[mid].u0_t : p.prob[mid].u0_w;
    if (s <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// The bf16 NF4 levels as byte planes for nf4_decode_word (scale 1).
__device__ __forceinline__ Nf4Table dc_level_table() { return nf4_table(1.0f); }

// X fragment of chunk c (16 k at k0 + 16 c) for token group tg: b0 = X[tok][k + 4q .. +1], b1 = X[tok][k + 4q + 2 .. +3].
__device__ __forceinline__ uint2 dc_xfrag(const DcProb& pr, int tok, int kk) {
  if (tok >= pr.m) return make_uint2(0u, 0u);
  return ldg_nc_v2(pr.x + static_cast<int64_t>(tok) * pr.k + kk);
}

template <int NG>
__global__ void __launch_bounds__(kDcThreads, 1) k_decode(const __grid_constant__ DcParams p) {
  __shared__ __align__(16) uint8_t s_ring[kDcWarps][kDcRing][kDcStage];
  __shared__ int s_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const long long u_begin = dc_run_start(blockIdx.x, p.units, p.grid);
  const long long u_end = dc_run_start(blockIdx.x + 1, p.units, p.grid);

  // ---------------------------------------------------------------- L2 prefetch of this run's bytes
  for (long long u = u_begin; u < u_end; ++u) {
    const bool tu = u < p.prob[0].u0_w;
    const DcProb& pr = p.prob[dc_find_prob(p, u, tu)];
    if (tu) {
      const int k0 = static_cast<int>(u - pr.u0_t) * pr.t_sub * kDcTChunk;
      const int kn = min(pr.t_sub * kDcTChunk, pr.k - k0);
      for (int j = threadIdx.x; j < pr.r; j += kDcThreads)
        prefetch_l2_bulk(pr.a + static_cast<int64_t>(j) * pr.k + k0, static_cast<uint32_t>(kn) * 2);
    } else {
      const long long w = u - pr.u0_w;
      const int tile = static_cast<int>(w / pr.ku), kun = static_cast<int>(w % pr.ku);
      for (int i = threadIdx.x; i < kDcRows; i += kDcThreads) {
        const int row = tile * kDcRows + i;
        if (row < pr.n) {
          prefetch_l2_bulk(pr.codes + static_cast<int64_t>(row) * (pr.k / 2) + kun * 128, 128);
          prefetch_l2_line(pr.absq + static_cast<int64_t>(row) * (pr.k / 64) + kun * kDcUnitBlocks);
        }
      }
    }
  }
  // X, sT, the counters and the workspace may come from earlier kernels of the stream
  griddep_wait();
  griddep_launch_dependents();

  const Nf4Table lv = dc_level_table();
  bool alive = true;

  // ---------------------------------------------------------------- T units
  long long u = u_begin;
  for (; u < u_end && u < p.prob[0].u0_w && alive; ++u) {
    const int pi = dc_find_prob(p, u, true);
    const DcProb& pr = p.prob[pi];
    const int tu = static_cast<int>(u - pr.u0_t);
    const int k0 = tu * pr.t_sub * kDcTChunk;
    const int kend = min(pr.k, k0 + pr.t_sub * kDcTChunk);
    // warp w: LoRA rows j = 16 w .. 16 w + 15 (r <= 128)
    float acc[NG][4];
#pragma unroll
    for (int t = 0; t < NG; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    const int j0 = warp * 16 + g, j1 = j0 + 8;
    if (warp * 16 < pr.r) {
      for (int kk = k0; kk < kend; kk += 16) {
        const int kq = kk + 4 * q;
        const uint2 a0 = j0 < pr.r ? ldg_nc_v2(pr.a + static_cast<int64_t>(j0) * pr.k + kq) : make_uint2(0u, 0u);
        const uint2 a1 = j1 < pr.r ? ldg_nc_v2(pr.a + static_cast<int64_t>(j1) * pr.k + kq) : make_uint2(0u, 0u);
#pragma unroll
        for (int t = 0; t < NG; ++t) {
          const uint2 xb = dc_xfrag(pr, t * 8 + g, kq);
          dc_mma(acc[t], a0.x, a1.x, a0.y, a1.y, xb.x, xb.y);
        }
      }
      // d[0] = (row j0, token 2q), d[1] = (j0, 2q+1), d[2] = (j1, 2q), d[3] = (j1, 2q+1)
      float* part = pr.tpart + static_cast<int64_t>(tu) * 16 * pr.r;
#pragma unroll
      for (int t = 0; t < NG; ++t) {
        const int tk = t * 8 + 2 * q;
        if (j0 < pr.r) {
          part[tk * pr.r + j0] = acc[t][0];
          part[(tk + 1) * pr.r + j0] = acc[t][1];
        }
        if (j1 < pr.r) {
          part[tk * pr.r + j1] = acc[t][2];
          part[(tk + 1) * pr.r + j1] = acc[t][3];
        }
      }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_flag = dc_arrive(pr.cnt, p.epoch) == static_cast<uint32_t>(pr.t_units);
    __syncthreads();
    if (s_flag) {
      // last T unit of the problem: T = sum of the partials in unit order -> t_save, sT
      __threadfence();
      for (int i = threadIdx.x; i < 16 * pr.r; i += kDcThreads) {
        const int tok = i / pr.r, j = i % pr.r;
        float v = 0.f;
        for (int c = 0; c < pr.t_units; ++c) v += __ldcg(pr.tpart + (static_cast<int64_t>(c) * 16 + tok) * pr.r + j);
        if (tok < pr.m && pr.t_save) pr.t_save[tok * pr.r + j] = v;
        pr.st[tok * pr.r + j] = __float2bfloat16_rn(tok < pr.m ? __fmul_rn(v, pr.scale) : 0.f);
      }
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) atomicAdd(pr.cnt, 1ull);  // count = t_units + 1: sT published
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- W units
  if (u >= u_end || !alive) return;
  // the run's (problem, tile, block) steps, walked twice: by the cp.async producer (ahead) and the consumer
  struct Cursor {
    long long u;
    int kb;  // block within the unit
  };
  const uint32_t ring0 = smem_u32(&s_ring[warp][0][0]);
  // stage block step `cur` of this warp's 16 rows into ring slot `slot`
  auto stage = [&](const Cursor& cur, int slot) {
    const int pi = dc_find_prob(p, cur.u, false);
    const DcProb& pr = p.prob[pi];
    const long long w = cur.u - pr.u0_w;
    const int tile = static_cast<int>(w / pr.ku), kun = static_cast<int>(w % pr.ku);
    const int row = tile * kDcRows + warp * 16 + (lane >> 1);
    const int kb = kun * kDcUnitBlocks + cur.kb;
    const bool ok = row < pr.n;
    const uint8_t* src = pr.codes + (ok ? static_cast<int64_t>(row) * (pr.k / 2) + kb * 32 + (lane & 1) * 16 : 0);
    cp_async16(ring0 + slot * kDcStage + (lane >> 1) * kDcPitch + (lane & 1) * 16, src, ok);
  };
  auto advance = [&](Cursor& cur) {
    if (++cur.kb == kDcUnitBlocks) {
      cur.kb = 0;
      ++cur.u;
    }
  };
  Cursor pre{u, 0};
  int issued = 0;
  for (; issued < kDcRing - 1; ++issued) {
    if (pre.u < u_end) {
      stage(pre, issued % kDcRing);
      advance(pre);
    }
    cp_async_commit();
  }

  float run[NG][4];
  auto zero_run = [&]() {
#pragma unroll
    for (int t = 0; t < NG; ++t) run[t][0] = run[t][1] = run[t][2] = run[t][3] = 0.f;
  };
  zero_run();
  int cur_pi = -1, cur_tile = -1;
  long long seg_first = u;  // first unit of the current segment

  // Finish the segment of tile (pi, tile) that ends at unit `seg_last`.
  auto flush = [&](int pi, int tile, long long seg_last) {
    const DcProb& pr = p.prob[pi];
    const long long tu0 = pr.u0_w + static_cast<long long>(tile) * pr.ku;  // first unit of the tile
    const long long tu1 = tu0 + pr.ku - 1;
    const int c0 = dc_cta_of(tu0, p.units, p.grid), c1 = dc_cta_of(tu1, p.units, p.grid);
    const int nseg = c1 - c0 + 1, seg = static_cast<int>(blockIdx.x) - c0;
    const int rbase = tile * kDcRows + warp * 16;
    float* slot = pr.ypart + (static_cast<int64_t>(tile) * p.maxseg) * 16 * kDcRows;
    float vals[NG][4];
    bool finalise = true;
    if (nseg > 1) {
      // C fragment: d[0] = (row g, tok 2q), d[1] = (g, 2q+1), d[2] = (g+8, 2q), d[3] = (g+8, 2q+1)
      float* mine = slot + static_cast<int64_t>(seg) * 16 * kDcRows;
#pragma unroll
      for (int t = 0; t < NG; ++t) {
        const int tk = t * 8 + 2 * q, rr = warp * 16 + g;
        mine[tk * kDcRows + rr] = run[t][0];
        mine[(tk + 1) * kDcRows + rr] = run[t][1];
        mine[tk * kDcRows + rr + 8] = run[t][2];
        mine[(tk + 1) * kDcRows + rr + 8] = run[t][3];
      }
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) s_flag = dc_arrive(pr.cnt + 2 + tile, p.epoch) == static_cast<uint32_t>(nseg);
      __syncthreads();
      finalise = s_flag != 0;
      if (finalise) {
        __threadfence();
#pragma unroll
        for (int t = 0; t < NG; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) vals[t][e] = 0.f;
        for (int sgi = 0; sgi < nseg; ++sgi) {
          const float* ps = slot + static_cast<int64_t>(sgi) * 16 * kDcRows;
#pragma unroll
          for (int t = 0; t < NG; ++t) {
            const int tk = t * 8 + 2 * q, rr = warp * 16 + g;
            vals[t][0] += __ldcg(ps + tk * kDcRows + rr);
            vals[t][1] += __ldcg(ps + (tk + 1) * kDcRows + rr);
            vals[t][2] += __ldcg(ps + tk * kDcRows + rr + 8);
            vals[t][3] += __ldcg(ps + (tk + 1) * kDcRows + rr + 8);
          }
        }
        if (threadIdx.x == 0) *reinterpret_cast<volatile unsigned long long*>(pr.cnt + 2 + tile) =
            static_cast<unsigned long long>(p.epoch) << 32;
      }
    } else {
#pragma unroll
      for (int t = 0; t < NG; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) vals[t][e] = run[t][e];
    }
    (void)seg_last;
    if (!finalise) return;
    // wait until the problem's sT is published (count t_units + 1)
    if (threadIdx.x == 0) {
      const unsigned long long want = (static_cast<unsigned long long>(p.epoch) << 32) | (pr.t_units + 1u);
      bool ok = *reinterpret_cast<volatile unsigned long long*>(pr.cnt) == want;
      if (!ok) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1;; ++it) {
          if (*reinterpret_cast<volatile unsigned long long*>(pr.cnt) == want) { ok = true; break; }
          if ((it & 63u) == 0 && globaltimer_ns() - t0 > p.wait_ns) break;
          __nanosleep(64);
        }
      }
      s_flag = ok;
      if (!ok) latch_status(p.status, ST_TIMEOUT);
    }
    __syncthreads();
    if (!s_flag) { alive = false; return; }
    __threadfence();
    // y = vals + sum_j sT[tok][j] B[row][j]
    const int rows[2] = {rbase + g, rbase + g + 8};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = rows[h];
      if (row >= pr.n) continue;
      const __nv_bfloat16* brow = pr.b + static_cast<int64_t>(row) * pr.r;
#pragma unroll
      for (int t = 0; t < NG; ++t) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = t * 8 + 2 * q + e;
          if (tok >= pr.m) continue;
          float v = vals[t][2 * h + e];
          const __nv_bfloat16* srow = pr.st + tok * pr.r;
          float l = 0.f;
          for (int j = 0; j < pr.r; ++j)
            l = fmaf(__bfloat162float(__ldcg(srow + j)), __bfloat162float(brow[j]), l);
          pr.y[static_cast<int64_t>(tok) * pr.n + row] = __float2bfloat16_rn(v + l);
        }
      }
    }
    // the problem's last tile returns its T and tiles-done counters to (epoch, 0)
    __syncthreads();
    if (threadIdx.x == 0 && dc_arrive(pr.cnt + 1, p.epoch) == static_cast<uint32_t>(pr.tiles)) {
      *reinterpret_cast<volatile unsigned long long*>(pr.cnt) = static_cast<unsigned long long>(p.epoch) << 32;
      *reinterpret_cast<volatile unsigned long long*>(pr.cnt + 1) = static_cast<unsigned long long>(p.epoch) << 32;
    }
  };

  Cursor cur{u, 0};
  const uint32_t pick = (q & 1) ? 0x7632u : 0x5410u;  // the two code bytes of chunk c in the 32-bit word
  float blk[NG][4];
  while (cur.u < u_end && alive) {
    const int pi = dc_find_prob(p, cur.u, false);
    const DcProb& pr = p.prob[pi];
    const long long w = cur.u - pr.u0_w;
    const int tile = static_cast<int>(w / pr.ku), kun = static_cast<int>(w % pr.ku);
    if (pi != cur_pi || tile != cur_tile) {
      if (cur_pi >= 0) {
        flush(cur_pi, cur_tile, cur.u - 1);
        if (!alive) break;
      }
      cur_pi = pi;
      cur_tile = tile;
      seg_first = cur.u;
      zero_run();
    }
    // keep the ring kDcRing - 1 blocks ahead
    if (pre.u < u_end) {
      stage(pre, issued % kDcRing);
      advance(pre);
    }
    cp_async_commit();
    ++issued;
    cp_async_wait<kDcRing - 1>();
    __syncwarp();
    const int slot = (issued - kDcRing) % kDcRing;
    const int kb = kun * kDcUnitBlocks + cur.kb;
    const int row0 = tile * kDcRows + warp * 16 + g, row1 = row0 + 8;
    const int kbr = pr.k / 64;
    // restored block scales of rows g, g + 8
    const float mu = *pr.mean;
    float a2[2] = {0.f, 0.f};
    if (row0 < pr.n) {
      const int64_t bi = static_cast<int64_t>(row0) * kbr + kb;
      a2[0] = restore_absmax(pr.absq[bi], pr.step[bi >> 8], mu);
    }
    if (row1 < pr.n) {
      const int64_t bi = static_cast<int64_t>(row1) * kbr + kb;
      a2[1] = restore_absmax(pr.absq[bi], pr.step[bi >> 8], mu);
    }
    const uint8_t* st0 = &s_ring[warp][slot][0];
    const uint4 c0a = *reinterpret_cast<const uint4*>(st0 + g * kDcPitch);
    const uint4 c0b = *reinterpret_cast<const uint4*>(st0 + g * kDcPitch + 16);
    const uint4 c1a = *reinterpret_cast<const uint4*>(st0 + (g + 8) * kDcPitch);
    const uint4 c1b = *reinterpret_cast<const uint4*>(st0 + (g + 8) * kDcPitch + 16);
    // chunk c (16 k) uses code bytes 8c + 2q, 8c + 2q + 1 of the 32-byte block; a word of
    // chunks (c, c+1) = bytes (8c + 2q, +1, 8c + 8 + 2q, +1)
    const uint32_t r0w[8] = {c0a.x, c0a.y, c0a.z, c0a.w, c0b.x, c0b.y, c0b.z, c0b.w};
    const uint32_t r1w[8] = {c1a.x, c1a.y, c1a.z, c1a.w, c1b.x, c1b.y, c1b.z, c1b.w};
#pragma unroll
    for (int t = 0; t < NG; ++t) blk[t][0] = blk[t][1] = blk[t][2] = blk[t][3] = 0.f;
    const int kbase = kb * 64;
#pragma unroll
    for (int cp = 0; cp < 2; ++cp) {  // chunk pairs (0,1), (2,3)
      const int wi = 4 * cp + (q >> 1);
      const uint32_t w0 = prmt(r0w[wi], r0w[wi + 2], pick);
      const uint32_t w1 = prmt(r1w[wi], r1w[wi + 2], pick);
      uint32_t d0[4], d1[4];
      nf4_decode_word(lv, w0, d0);
      nf4_decode_word(lv, w1, d1);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = 2 * cp + h;
        const int kq = kbase + 16 * c + 4 * q;
#pragma unroll
        for (int t = 0; t < NG; ++t) {
          const uint2 xb = dc_xfrag(pr, t * 8 + g, kq);
          dc_mma(blk[t], d0[2 * h], d1[2 * h], d0[2 * h + 1], d1[2 * h + 1], xb.x, xb.y);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < NG; ++t) {
      run[t][0] = fmaf(a2[0], blk[t][0], run[t][0]);
      run[t][1] = fmaf(a2[0], blk[t][1], run[t][1]);
      run[t][2] = fmaf(a2[1], blk[t][2], run[t][2]);
      run[t][3] = fmaf(a2[1], blk[t][3], run[t][3]);
    }
    __syncwarp();  // the slot is refilled by a later stage()
    advance(cur);
  }
  cp_async_wait<0>();
  if (cur_pi >= 0 && alive) flush(cur_pi, cur_tile, cur.u - 1);
  (void)seg_first;
}

// ---------------------------------------------------------------------------- host
int decode_max_problems() { return kDcMaxProbs; }

namespace {
struct DcPlan {
  int grid, maxseg;
  long long units;
  size_t ws_bytes;
  std::vector<size_t> off_cnt, off_tpart, off_st, off_ypart;
  std::vector<int> t_units, t_sub, tiles, ku, u0_t, u0_w;
};

size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

DcPlan dc_plan(const GroupedProblem* probs, int count, int num_sms) {
  DcPlan pl;
  pl.grid = num_sms > 0 ? num_sms : 1;
  pl.t_units.resize(count);
  pl.t_sub.resize(count);
  pl.tiles.resize(count);
  pl.ku.resize(count);
  pl.u0_t.resize(count);
  pl.u0_w.resize(count);
  long long u = 0;
  for (int i = 0; i < count; ++i) {
    const int kc = static_cast<int>(probs[i].w.k / kDcTChunk);  // k % 64 == 0, k >= 64
    const int kchunks = kc > 0 ? kc : 1;
    pl.t_sub[i] = (kchunks + 7) / 8;  // about 8 T units per problem
    pl.t_units[i] = (kchunks + pl.t_sub[i] - 1) / pl.t_sub[i];
    if (static_cast<long long>(pl.t_units[i]) * pl.t_sub[i] * kDcTChunk < probs[i].w.k) ++pl.t_units[i];
    pl.u0_t[i] = static_cast<int>(u);
    u += pl.t_units[i];
  }
  for (int i = 0; i < count; ++i) {
    pl.tiles[i] = static_cast<int>((probs[i].w.n + kDcRows - 1) / kDcRows);
    pl.ku[i] = static_cast<int>((probs[i].w.k + 255) / 256);
    pl.u0_w[i] = static_cast<int>(u);
    u += static_cast<long long>(pl.tiles[i]) * pl.ku[i];
  }
  pl.units = u;
  if (pl.grid > u) pl.grid = static_cast<int>(u);
  // the most runs any tile is split over
  auto cta_of = [&](long long uu) { return static_cast<int>(((uu + 1) * pl.grid - 1) / pl.units); };
  pl.maxseg = 1;
  for (int i = 0; i < count; ++i)
    for (int t = 0; t < pl.tiles[i]; ++t) {
      const long long a = pl.u0_w[i] + static_cast<long long>(t) * pl.ku[i];
      const int s = cta_of(a + pl.ku[i] - 1) - cta_of(a) + 1;
      if (s > pl.maxseg) pl.maxseg = s;
    }
  size_t off = 0;
  pl.off_cnt.resize(count);
  pl.off_tpart.resize(count);
  pl.off_st.resize(count);
  pl.off_ypart.resize(count);
  for (int i = 0; i < count; ++i) {
    pl.off_cnt[i] = off;
    off += al256(static_cast<size_t>(2 + pl.tiles[i]) * 8);
    pl.off_tpart[i] = off;
    off += al256(static_cast<size_t>(pl.t_units[i]) * 16 * probs[i].r * 4);
    pl.off_st[i] = off;
    off += al256(static_cast<size_t>(16) * probs[i].r * 2);
    pl.off_ypart[i] = off;
    off += al256(static_cast<size_t>(pl.tiles[i]) * pl.maxseg * 16 * kDcRows * 4);
  }
  pl.ws_bytes = off;
  return pl;
}
}  // namespace

size_t decode_workspace_bytes(const GroupedProblem* probs, int count, int num_sms) {
  return dc_plan(probs, count, num_sms).ws_bytes;
}

cudaError_t launch_decode(const GroupedProblem* probs, int count, void* ws, uint32_t epoch, unsigned* status,
                          uint64_t wait_ns, int num_sms, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  const DcPlan pl = dc_plan(probs, count, num_sms);
  static DcParams prm;  // 20+ KB: not on the host stack; launches copy it
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  prm.count = count;
  prm.grid = pl.grid;
  prm.maxseg = pl.maxseg;
  prm.epoch = epoch;
  prm.units = pl.units;
  prm.wait_ns = wait_ns;
  prm.status = status;
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
    d.st = reinterpret_cast<__nv_bfloat16*>(base + pl.off_st[i]);
    d.ypart = reinterpret_cast<float*>(base + pl.off_ypart[i]);
    d.cnt = reinterpret_cast<unsigned long long*>(base + pl.off_cnt[i]);
    d.n = static_cast<int>(g.w.n);
    d.k = static_cast<int>(g.w.k);
    d.m = g.m;
    d.r = g.r;
    d.scale = g.alpha / static_cast<float>(g.r);
    d.t_units = pl.t_units[i];
    d.t_sub = pl.t_sub[i];
    d.tiles = pl.tiles[i];
    d.ku = pl.ku[i];
    d.u0_t = pl.u0_t[i];
    d.u0_w = pl.u0_w[i];
    if (g.m > mmax) mmax = g.m;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kDcThreads);
  cfg.dynamicSmemBytes = 0;
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
