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
// prefetches (one plain prefetch per 128-byte line) for the code bytes it will read first -- the weights do not depend on
// the previous kernel -- and only then waits (griddepcontrol.wait) for the
// preceding kernel of the stream; right after that wait it lets the next
// kernel launch, which prefetches its own weights while this one computes.
//
// Work: first, X A^T is cut into about one k-slice per CTA (slice i on CTA
// i % grid, the 8 warps splitting its 16-k chunks); the last slice of a
// problem adds the slices' partials in slice order and publishes
// sT = bf16(s X A^T).  Then the weights are cut into W units of equal size
// (problem, tile of 128 rows, 256 k) and every CTA (two per SM) takes one
// contiguous run of them.  A run accumulates the units of one row tile in
// registers; a tile split between runs leaves float32 partials that the last
// arriving CTA adds in run order (deterministic).  The tile's finaliser adds
// the LoRA term with sT; a finaliser that gets there first waits for it
// (bounded wait; every CTA of the grid is resident: the grid has at most one
// CTA per SM and the next kernel can only launch after every CTA of this one
// has started).
//
// A W unit: warp w owns rows 16w .. 16w+15 of the tile; per 64-wide absmax
// block, lanes stage the 16 rows x 32 code bytes into a shared-memory ring with
// cp.async (kDcRing blocks ahead; the block scales are loaded two blocks
// ahead, the X fragments before the decode), decode them with the byte-permute table of
// the bf16 NF4 levels into mma.sync m16n8k16 A fragments (k permuted so lane
// (g, q) holds k = 16c + 4q .. 4q+3 of chunk c), and multiply with the X
// fragments (8 tokens per MMA, 1 or 2 groups) into a per-block accumulator,
// which is scaled by the block's restored scale a' and added to the run's sum.
// So the effective weight is bf16(L[code]) * a' with a' applied in float32 to
// the block's partial sums (within 2^-8 relative of the bf16_rn(L a') the
// fwd/bwd GEMMs use).
//
// Counters are plain words updated with one atomic add each (many CTAs arrive
// on the same word, so no retry loops); every counter is returned to zero by
// its last user, so a workspace that starts zeroed stays zeroed across calls
// and graph replays.
#include <algorithm>
#include <cstdio>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kDcWarps = 8;
constexpr int kDcCtasPerSm = 2;            // two CTAs (16 warps) per SM hide the decode's latency
constexpr int kDcThreads = kDcWarps * 32;
constexpr int kDcRows = kDcWarps * 16;     // rows per tile
constexpr int kDcUnitBlocks = 4;           // 64-wide blocks per W unit (256 k)
constexpr int kDcRing = 6;                 // cp.async ring depth per warp, in blocks
constexpr int kDcPitch = 48;               // shared-memory bytes per staged row piece (32 used, padded: no bank conflicts)
constexpr int kDcStage = 16 * kDcPitch;    // one block of the warp's 16 rows
constexpr int kDcMaxProbs = 128;
constexpr int kDcPrefetchUnits = 24;
constexpr int kDcMaxSlices = 16;           // X A^T slices per problem (each finaliser adds them all)       // W units a CTA keeps prefetched into L2 ahead of its consumer

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
  float* ypart;             // [tiles][maxseg][16][128] partial Y
  unsigned* cnt;            // [2 + tiles]: T, tiles done, then one per tile (zero between calls)
  int n, k, m, r;
  float scale;
  int t_slices, t_w, s0;    // X A^T: slices of t_w 64-wide blocks, first global slice
  int tiles, ku;            // row tiles, W units per tile (ceil(k / 256))
  long long u0_w;           // first W unit (global unit index)
};

struct DcParams {
  int count;
  int grid;
  int maxseg;
  long long units;            // W units of the call
  int slices;                 // X A^T slices of the call (slice i goes to CTA i % grid)
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
// The same load predicated in the instruction itself (zero when `on` is false; no branch).
__device__ __forceinline__ uint2 ldg_nc_v2_if(const void* p, bool on) {
  uint2 v = make_uint2(0u, 0u);
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q ld.global.nc.v2.u32 {%0,%1}, [%3];\n\t}"
      : "+r"(v.x), "+r"(v.y)
      : "r"(static_cast<int>(on)), "l"(p));
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

__device__ __forceinline__ void prefetch_l2_line(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// L2 prefetch of `bytes` bytes from p: one plain prefetch per 128-byte line touched (regular
// memory instructions: a warp covers 32 lines per instruction, unlike one bulk copy per row).
__device__ __forceinline__ void dc_prefetch_codes(const void* p, int bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(127);
  const uintptr_t a1 = reinterpret_cast<uintptr_t>(p) + bytes;
  for (uintptr_t a = a0; a < a1; a += 128) prefetch_l2_line(reinterpret_cast<const void*>(a));
}

// First unit of CTA c when `units` units are dealt to `grid` CTAs in contiguous runs.
__device__ __forceinline__ long long dc_run_start(int c, long long units, int grid) {
  return static_cast<long long>(c) * units / grid;
}
// CTA whose run holds unit u.
__device__ __forceinline__ int dc_cta_of(long long u, long long units, int grid) {
  return static_cast<int>(((u + 1) * grid - 1) / units);
}

// Arrive on a counter (one atomic, no retry loop: many CTAs arrive on the same word); returns
// the count after this arrival.  Every counter is returned to zero by its last user.
__device__ __forceinline__ uint32_t dc_arrive(unsigned* c) { return atomicAdd(c, 1u) + 1u; }

__device__ __forceinline__ int dc_find_prob(const DcParams& p, long long u) {  // problem of W unit u
  int lo = 0, hi = p.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.prob[mid].u0_w <= u) lo = mid; else hi = mid - 1;
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

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
// Decode one 32-bit word of packed codes (byte b: element 2b in the high nibble, 2b+1 in the low)
// into 4 bf16x2 words (element 2i in the low half of out[i]) through this lane's column of the
// level-pair table (row stride 128 bytes).
__device__ __forceinline__ void dc_decode_word(uint32_t lut_lane, uint32_t w, uint32_t (&out)[4]) {
  out[0] = lds32(lut_lane + ((w << 7) & 0x7f80u));
  out[1] = lds32(lut_lane + ((w >> 1) & 0x7f80u));
  out[2] = lds32(lut_lane + ((w >> 9) & 0x7f80u));
  out[3] = lds32(lut_lane + ((w >> 17) & 0x7f80u));
}

// Four bf16 values row[j .. j+3] of a row of length r (zero past r) as two bf16x2 words.
// `readonly`: the row is not written during the kernel (non-coherent path); otherwise it is read
// through L2 (sT, written by another CTA of this grid).
__device__ __forceinline__ uint2 dc_ld_bf16x4(const __nv_bfloat16* row, int j, int r, bool readonly) {
  if ((r & 3) == 0 && j + 4 <= r) {  // 8-byte aligned: rows of r % 4 == 0 values, j % 4 == 0
    if (readonly) return ldg_nc_v2(row + j);
    return __ldcg(reinterpret_cast<const uint2*>(row + j));
  }
  const unsigned short* u = reinterpret_cast<const unsigned short*>(row);
  uint32_t v[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) v[e] = j + e < r ? (readonly ? __ldg(u + j + e) : __ldcg(u + j + e)) : 0u;
  return make_uint2(v[0] | (v[1] << 16), v[2] | (v[3] << 16));
}

// X fragment of chunk c (16 k at k0 + 16 c) for token group tg: b0 = X[tok][k + 4q .. +1], b1 = X[tok][k + 4q + 2 .. +3].
__device__ __forceinline__ uint2 dc_xfrag(const DcProb& pr, int tok, int kk) {
  if (tok >= pr.m) return make_uint2(0u, 0u);
  return ldg_nc_v2(pr.x + static_cast<int64_t>(tok) * pr.k + kk);
}

template <int NG>
__global__ void __launch_bounds__(kDcThreads, kDcCtasPerSm) k_decode(const __grid_constant__ DcParams p) {
  __shared__ __align__(16) uint8_t s_ring[kDcWarps][kDcRing][kDcStage];
  __shared__ float s_red[kDcWarps][16][16];
  __shared__ int s_flag;
  // level pairs of a code byte: s_lut[b * 32 + lane] = bf16 L[b >> 4] | (bf16 L[b & 15]) << 16, the
  // byte's two weights in mma fragment order; one column per lane, so lookups never conflict
  extern __shared__ __align__(16) uint32_t s_lut[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const long long u_begin = dc_run_start(blockIdx.x, p.units, p.grid);
  const long long u_end = dc_run_start(blockIdx.x + 1, p.units, p.grid);

  // ---------------------------------------------------------------- L2 prefetch (before the wait)
  // the first kDcPrefetchUnits W units of this run (every unit's codes when the call is a decoder
  // stage; later units of long lists are prefetched as the run advances) and this CTA's T slices
  for (long long u = u_begin; u < u_end && u < u_begin + kDcPrefetchUnits; ++u) {
    const DcProb& pr = p.prob[dc_find_prob(p, u)];
    const long long w = u - pr.u0_w;
    const int tile = static_cast<int>(w / pr.ku), kun = static_cast<int>(w % pr.ku);
    const int nb = min(kDcUnitBlocks, pr.k / 64 - kun * kDcUnitBlocks);  // the last unit of a row may be short
    for (int i = threadIdx.x; i < kDcRows; i += kDcThreads) {
      const int row = tile * kDcRows + i;
      if (row < pr.n) {
        dc_prefetch_codes(pr.codes + static_cast<int64_t>(row) * (pr.k / 2) + kun * 128, nb * 32);
        prefetch_l2_line(pr.absq + static_cast<int64_t>(row) * (pr.k / 64) + kun * kDcUnitBlocks);
      }
    }
  }
  for (int sl = blockIdx.x; sl < p.slices; sl += p.grid) {
    const DcProb& pr = p.prob[dc_find_slice(p, sl)];
    const int kb0 = (sl - pr.s0) * pr.t_w, kb1 = min(pr.k / 64, kb0 + pr.t_w);
    for (int j = threadIdx.x; j < pr.r; j += kDcThreads)
      dc_prefetch_codes(pr.a + static_cast<int64_t>(j) * pr.k + kb0 * 64, (kb1 - kb0) * 128);
  }
  {
    // the 16 bf16 levels go through shared memory (a dynamically indexed local array would put
    // the whole kernel on a stack frame)
    __shared__ uint32_t s_lv[16];
    if (threadIdx.x < 16) {
      constexpr uint32_t hex[16] = QLORA_NF4_LEVELS_HEX;
      uint32_t v = 0;
#pragma unroll
      for (int c = 0; c < 16; ++c) v = threadIdx.x == c ? hex[c] : v;
      s_lv[threadIdx.x] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v)));
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 256 * 32; i += kDcThreads) {
      const int b = i >> 5;
      s_lut[i] = s_lv[b >> 4] | (s_lv[b & 15] << 16);
    }
    __syncthreads();  // a CTA with no T slice reads the table next
  }
  // X, sT, the counters and the workspace may come from earlier kernels of the stream
  griddep_wait();
  griddep_launch_dependents();

  // ---------------------------------------------------------------- T = X A^T, spread over every CTA
  // slice sl (problem p, 64-wide blocks [kb0, kb1)) goes to CTA sl % grid; the 8 warps split its
  // 16-k chunks, the CTA adds their partial sums in warp order into the slice's partial
  for (int sl = blockIdx.x; sl < p.slices; sl += p.grid) {
    const DcProb& pr = p.prob[dc_find_slice(p, sl)];
    const int si = sl - pr.s0;
    const int kb0 = si * pr.t_w, kb1 = min(pr.k / 64, kb0 + pr.t_w);
    const int nch = (kb1 - kb0) * 4;
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
          const uint2 xb = dc_xfrag(pr, t * 8 + g, kq);
          dc_mma(acc[t], a0.x, a1.x, a0.y, a1.y, xb.x, xb.y);
        }
      }
      // C fragment: d[0] = (row j0, tok 2q), d[1] = (j0, 2q+1), d[2] = (j1, 2q), d[3] = (j1, 2q+1)
#pragma unroll
      for (int t = 0; t < NG; ++t) {
        const int tk = t * 8 + 2 * q;
        s_red[warp][tk][g] = acc[t][0];
        s_red[warp][tk + 1][g] = acc[t][1];
        s_red[warp][tk][g + 8] = acc[t][2];
        s_red[warp][tk + 1][g + 8] = acc[t][3];
      }
      __syncthreads();
      {
        const int tok = threadIdx.x >> 4, j = threadIdx.x & 15;  // 256 threads = 16 tokens x 16 j
        if (tok < NG * 8 && jg * 16 + j < pr.r) {
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kDcWarps; ++w) v += s_red[w][tok][j];
          pr.tpart[(static_cast<int64_t>(si) * 16 + tok) * pr.r + jg * 16 + j] = v;
        }
      }
      __syncthreads();
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) dc_arrive(pr.cnt);  // count == t_slices: every slice partial of the problem is written
  }

  // ---------------------------------------------------------------- W units
  if (u_begin >= u_end) return;
  // A unit's place: problem, row tile, 256-k unit within the tile, blocks in the unit.  Found by a
  // binary search and one division at the start of the run; after that the cursors step (the
  // units of a run are consecutive: k units of a tile, then the next tile, then the next problem).
  struct Unit {
    int pi, tile, kun, nb;  // nb: blocks in the unit (the last unit of a row may hold fewer than 4)
  };
  auto unit_nb = [&](const Unit& d) { return min(kDcUnitBlocks, p.prob[d.pi].k / 64 - d.kun * kDcUnitBlocks); };
  auto describe = [&](long long uu) {
    Unit d;
    d.pi = dc_find_prob(p, uu);
    const DcProb& pr = p.prob[d.pi];
    const int w = static_cast<int>(uu - pr.u0_w);
    d.tile = w / pr.ku;
    d.kun = w - d.tile * pr.ku;
    d.nb = unit_nb(d);
    return d;
  };
  auto step_unit = [&](Unit& d) {
    if (++d.kun == p.prob[d.pi].ku) {
      d.kun = 0;
      if (++d.tile == p.prob[d.pi].tiles) {
        d.tile = 0;
        if (d.pi + 1 < p.count) ++d.pi;
      }
    }
    d.nb = unit_nb(d);
  };
  // ---- the cp.async stager: runs kDcRing - 1 blocks ahead of the consumer through the run
  const uint32_t stage_dst0 = smem_u32(&s_ring[warp][0][0]) + (lane >> 1) * kDcPitch + (lane & 1) * 16;
  long long st_u = u_begin;
  int st_kb = 0, st_slot = 0;
  int st_left = static_cast<int>(u_end - u_begin);  // units the stager has not finished
  Unit st_d = describe(u_begin);
  const uint8_t* st_src = nullptr;
  bool st_ok = false;
  auto st_enter = [&]() {
    const DcProb& pr = p.prob[st_d.pi];
    const int row = st_d.tile * kDcRows + warp * 16 + (lane >> 1);
    st_ok = row < pr.n;
    st_src = pr.codes + (st_ok ? static_cast<int64_t>(row) * (pr.k / 2) + st_d.kun * 128 + (lane & 1) * 16 : 0);
    st_kb = 0;
  };
  auto stage_next = [&]() {
    if (st_left > 0) {
      cp_async16(stage_dst0 + st_slot * kDcStage, st_src, st_ok);
      st_src += 32;
      if (++st_kb == st_d.nb) {
        ++st_u;
        --st_left;
        step_unit(st_d);
        st_enter();
      }
    }
    cp_async_commit();
    st_slot = st_slot + 1 == kDcRing ? 0 : st_slot + 1;
  };
  st_enter();
  for (int i = 0; i < kDcRing - 1; ++i) stage_next();
  int use_slot = 0;

  // raw block scales of rows g, g+8 for the blocks of a unit, loaded one unit before use
  struct Scales {
    int q0[kDcUnitBlocks], q1[kDcUnitBlocks];
    float s0[kDcUnitBlocks], s1[kDcUnitBlocks];
    float mu;
  };
  auto load_scales = [&](const Unit& d, Scales& sc) {
    const DcProb& pr = p.prob[d.pi];
    const int kbr = pr.k / 64;
    const int r0 = d.tile * kDcRows + warp * 16 + g, r1 = r0 + 8;
    const int64_t b0 = static_cast<int64_t>(r0) * kbr + d.kun * kDcUnitBlocks;
    const int64_t b1 = b0 + static_cast<int64_t>(8) * kbr;
    sc.mu = __ldg(pr.mean);
#pragma unroll
    for (int b = 0; b < kDcUnitBlocks; ++b) {
      const bool in = b < d.nb;
      sc.q0[b] = (in && r0 < pr.n) ? __ldg(pr.absq + b0 + b) : 0;
      sc.s0[b] = (in && r0 < pr.n) ? __ldg(pr.step + ((b0 + b) >> 8)) : 0.f;
      sc.q1[b] = (in && r1 < pr.n) ? __ldg(pr.absq + b1 + b) : 0;
      sc.s1[b] = (in && r1 < pr.n) ? __ldg(pr.step + ((b1 + b) >> 8)) : 0.f;
    }
  };
  long long cu = u_begin;
  Unit cd = describe(cu);
  Scales sc_cur, sc_nxt;
  load_scales(cd, sc_cur);
  // the rolling L2 prefetch cursor, kDcPrefetchUnits units ahead of the consumer
  Unit pf_d = describe(u_begin + kDcPrefetchUnits < u_end ? u_begin + kDcPrefetchUnits : u_begin);

  float run[NG][4];
  auto zero_run = [&]() {
#pragma unroll
    for (int t = 0; t < NG; ++t) run[t][0] = run[t][1] = run[t][2] = run[t][3] = 0.f;
  };
  zero_run();
  int cur_pi = -1, cur_tile = -1;
  bool alive = true;

  // Finish this run's segment of tile (pi, tile): add the segments' partials when the tile is
  // split between runs (the last arriving run does it), then the LoRA term, then write y.
  auto flush = [&](int pi, int tile) {
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
      if (threadIdx.x == 0) s_flag = dc_arrive(pr.cnt + 2 + tile) == static_cast<uint32_t>(nseg);
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
        __syncthreads();
        if (threadIdx.x == 0) *reinterpret_cast<volatile unsigned*>(pr.cnt + 2 + tile) = 0u;
      }
    } else {
#pragma unroll
      for (int t = 0; t < NG; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) vals[t][e] = run[t][e];
    }
    if (!finalise) return;
    // wait until every X A^T slice of the problem is written (count == t_slices)
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
    if (!s_flag) { alive = false; return; }
    __threadfence();
    // sT = bf16(s X A^T) for this problem, the slices' partials added in slice order (every
    // finaliser of the problem adds the same values in the same order); the finaliser of tile 0
    // also writes t_save.  Kept in shared memory as bf16 pairs [16 tokens][64 pairs].
    uint32_t* s_st = reinterpret_cast<uint32_t*>(&s_red[0][0][0]);
    {
      const int rpad = (pr.r + 15) & ~15, hp = rpad / 2;
      const int64_t cstride = static_cast<int64_t>(16) * pr.r;
      for (int i = threadIdx.x; i < 16 * hp; i += kDcThreads) {
        const int tok = i / hp, jp = i % hp, j = 2 * jp;
        float v0 = 0.f, v1 = 0.f;
        if (tok < pr.m) {
          const float* src = pr.tpart + static_cast<int64_t>(tok) * pr.r + j;
          float x0[kDcMaxSlices], x1[kDcMaxSlices];
#pragma unroll
          for (int c = 0; c < kDcMaxSlices; ++c) {
            x0[c] = (c < pr.t_slices && j < pr.r) ? __ldcg(src + c * cstride) : 0.f;
            x1[c] = (c < pr.t_slices && j + 1 < pr.r) ? __ldcg(src + c * cstride + 1) : 0.f;
          }
#pragma unroll
          for (int c = 0; c < kDcMaxSlices; ++c) {
            v0 += x0[c];
            v1 += x1[c];
          }
          if (tile == 0 && pr.t_save) {
            if (j < pr.r) pr.t_save[tok * pr.r + j] = v0;
            if (j + 1 < pr.r) pr.t_save[tok * pr.r + j + 1] = v1;
          }
        }
        s_st[tok * 64 + jp] = tok < pr.m ? pack_bf16x2_rn(__fmul_rn(v0, pr.scale), __fmul_rn(v1, pr.scale)) : 0u;
      }
    }
    __syncthreads();
    // y = vals + sT B^T: the LoRA up-projection as extra 16-wide k chunks of the same MMA
    // (A = rows of B, k = j; B operand = sT [tok][j]), accumulated in float32
    const int row0 = rbase + g, row1 = row0 + 8;
    for (int j0 = 0; j0 < pr.r; j0 += 16) {
      const int jq = j0 + 4 * q;
      const uint2 b0 = row0 < pr.n ? dc_ld_bf16x4(pr.b + static_cast<int64_t>(row0) * pr.r, jq, pr.r, true)
                                   : make_uint2(0u, 0u);
      const uint2 b1 = row1 < pr.n ? dc_ld_bf16x4(pr.b + static_cast<int64_t>(row1) * pr.r, jq, pr.r, true)
                                   : make_uint2(0u, 0u);
#pragma unroll
      for (int t = 0; t < NG; ++t) {
        const uint32_t* sp = s_st + (t * 8 + g) * 64 + jq / 2;
        dc_mma(vals[t], b0.x, b1.x, b0.y, b1.y, sp[0], sp[1]);
      }
    }
    const int rows[2] = {row0, row1};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = rows[h];
      if (row >= pr.n) continue;
#pragma unroll
      for (int t = 0; t < NG; ++t)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = t * 8 + 2 * q + e;
          if (tok < pr.m) pr.y[static_cast<int64_t>(tok) * pr.n + row] = __float2bfloat16_rn(vals[t][2 * h + e]);
        }
    }
    // the problem's last tile returns its T and tiles-done counters to zero
    __syncthreads();
    if (threadIdx.x == 0 && dc_arrive(pr.cnt + 1) == static_cast<uint32_t>(pr.tiles)) {
      *reinterpret_cast<volatile unsigned*>(pr.cnt) = 0u;
      *reinterpret_cast<volatile unsigned*>(pr.cnt + 1) = 0u;
    }
  };

  __syncthreads();  // s_lut written
  const uint32_t lut = smem_u32(s_lut + lane);
  const uint32_t pick = (q & 1) ? 0x7632u : 0x5410u;  // the two code bytes of chunk c in the 32-bit word
  const uint32_t ring_row0 = smem_u32(&s_ring[warp][0][0]) + g * kDcPitch;
  float blk[NG][4];
  while (cu < u_end && alive) {
    const DcProb& pr = p.prob[cd.pi];
    if (cd.pi != cur_pi || cd.tile != cur_tile) {
      if (cur_pi >= 0) {
        flush(cur_pi, cur_tile);
        if (!alive) break;
      }
      cur_pi = cd.pi;
      cur_tile = cd.tile;
      zero_run();
    }
    // the next unit: its place, its block scales, and the L2 prefetch kDcPrefetchUnits ahead
    Unit nd = cd;
    step_unit(nd);
    if (cu + 1 < u_end) load_scales(nd, sc_nxt);
    if (cu + kDcPrefetchUnits < u_end) {
      if (lane < 16) {
        const DcProb& pf = p.prob[pf_d.pi];
        const int row = pf_d.tile * kDcRows + warp * 16 + lane;
        if (row < pf.n)
          dc_prefetch_codes(pf.codes + static_cast<int64_t>(row) * (pf.k / 2) + pf_d.kun * 128, pf_d.nb * 32);
      }
      step_unit(pf_d);
    }
    // this lane's token rows of X for the unit (tokens g and g + 8), chunk c at +16 c, block b at +64 b
    const int k0 = cd.kun * kDcUnitBlocks * 64 + 4 * q;
    const __nv_bfloat16* xp[NG];
    bool xon[NG];
#pragma unroll
    for (int t = 0; t < NG; ++t) {
      xon[t] = t * 8 + g < pr.m;  // rows of absent tokens read as zero (the pointer stays inside X)
      xp[t] = pr.x + static_cast<int64_t>(xon[t] ? t * 8 + g : 0) * pr.k + k0;
    }
#pragma unroll
    for (int b = 0; b < kDcUnitBlocks; ++b) {
      if (b >= cd.nb) break;
      uint2 xf[4][NG];
#pragma unroll
      for (int t = 0; t < NG; ++t)
#pragma unroll
        for (int c = 0; c < 4; ++c) xf[c][t] = ldg_nc_v2_if(xp[t] + b * 64 + 16 * c, xon[t]);
      stage_next();
      cp_async_wait<kDcRing - 1>();
      __syncwarp();
      const uint32_t rr = ring_row0 + use_slot * kDcStage;
      use_slot = use_slot + 1 == kDcRing ? 0 : use_slot + 1;
      // the code words this lane decodes: words 4cp + q/2 and 4cp + 2 + q/2 of rows g and g + 8
      const uint32_t wq = rr + 4 * (q >> 1);
      const uint32_t a00 = lds32(wq), a01 = lds32(wq + 8), a02 = lds32(wq + 16), a03 = lds32(wq + 24);
      const uint32_t a10 = lds32(wq + 8 * kDcPitch), a11 = lds32(wq + 8 * kDcPitch + 8);
      const uint32_t a12 = lds32(wq + 8 * kDcPitch + 16), a13 = lds32(wq + 8 * kDcPitch + 24);
#pragma unroll
      for (int t = 0; t < NG; ++t) blk[t][0] = blk[t][1] = blk[t][2] = blk[t][3] = 0.f;
#pragma unroll
      for (int cp = 0; cp < 2; ++cp) {  // chunk pairs (0,1), (2,3)
        const uint32_t w0 = prmt(cp ? a02 : a00, cp ? a03 : a01, pick);
        const uint32_t w1 = prmt(cp ? a12 : a10, cp ? a13 : a11, pick);
        uint32_t d0[4], d1[4];
        dc_decode_word(lut, w0, d0);
        dc_decode_word(lut, w1, d1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = 2 * cp + h;
#pragma unroll
          for (int t = 0; t < NG; ++t)
            dc_mma(blk[t], d0[2 * h], d1[2 * h], d0[2 * h + 1], d1[2 * h + 1], xf[c][t].x, xf[c][t].y);
        }
      }
      const float a20 = restore_absmax(static_cast<int8_t>(sc_cur.q0[b]), sc_cur.s0[b], sc_cur.mu);
      const float a21 = restore_absmax(static_cast<int8_t>(sc_cur.q1[b]), sc_cur.s1[b], sc_cur.mu);
#pragma unroll
      for (int t = 0; t < NG; ++t) {
        run[t][0] = fmaf(a20, blk[t][0], run[t][0]);
        run[t][1] = fmaf(a20, blk[t][1], run[t][1]);
        run[t][2] = fmaf(a21, blk[t][2], run[t][2]);
        run[t][3] = fmaf(a21, blk[t][3], run[t][3]);
      }
      __syncwarp();  // the slot is refilled by a later stage_next()
    }
    sc_cur = sc_nxt;
    cd = nd;
    ++cu;
  }
  cp_async_wait<0>();
  if (cur_pi >= 0 && alive) flush(cur_pi, cur_tile);
}

// ---------------------------------------------------------------------------- host
int decode_max_problems() { return kDcMaxProbs; }

namespace {
struct DcPlan {
  int grid, maxseg, slices;
  long long units;
  size_t ws_bytes;
  std::vector<size_t> off_cnt, off_tpart, off_ypart;
  std::vector<int> t_slices, t_w, s0, tiles, ku;
  std::vector<long long> u0_w;
};

size_t al256(size_t b) { return (b + 255) & ~size_t(255); }

DcPlan dc_plan(const GroupedProblem* probs, int count, int num_sms) {
  DcPlan pl;
  const int sms = num_sms > 0 ? num_sms : 1;
  pl.t_slices.resize(count);
  pl.t_w.resize(count);
  pl.s0.resize(count);
  pl.tiles.resize(count);
  pl.ku.resize(count);
  pl.u0_w.resize(count);
  // W units
  long long u = 0;
  for (int i = 0; i < count; ++i) {
    pl.tiles[i] = static_cast<int>((probs[i].w.n + kDcRows - 1) / kDcRows);
    pl.ku[i] = static_cast<int>((probs[i].w.k + 255) / 256);
    pl.u0_w[i] = u;
    u += static_cast<long long>(pl.tiles[i]) * pl.ku[i];
  }
  pl.units = u;
  const long long slots = static_cast<long long>(sms) * kDcCtasPerSm;  // every CTA of the grid resident at once
  pl.grid = static_cast<int>(u < slots ? u : slots);
  // X A^T slices: about one per CTA over the whole list, in proportion to each problem's r k
  double work = 0.0;
  for (int i = 0; i < count; ++i) work += static_cast<double>((probs[i].r + 15) / 16) * probs[i].w.k;
  int sl = 0;
  for (int i = 0; i < count; ++i) {
    const int blocks = static_cast<int>(probs[i].w.k / 64);
    const double share = static_cast<double>((probs[i].r + 15) / 16) * probs[i].w.k / work;
    int want = static_cast<int>(share * pl.grid + 0.5);
    want = want < 1 ? 1 : (want > blocks ? blocks : want);
    if (want > kDcMaxSlices) want = kDcMaxSlices;
    pl.t_w[i] = (blocks + want - 1) / want;
    pl.t_slices[i] = (blocks + pl.t_w[i] - 1) / pl.t_w[i];
    pl.s0[i] = sl;
    sl += pl.t_slices[i];
  }
  pl.slices = sl;
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
  pl.off_ypart.resize(count);
  for (int i = 0; i < count; ++i) {
    pl.off_cnt[i] = off;
    off += al256(static_cast<size_t>(2 + pl.tiles[i]) * 4);
    pl.off_tpart[i] = off;
    off += al256(static_cast<size_t>(pl.t_slices[i]) * 16 * probs[i].r * 4);
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

cudaError_t launch_decode(const GroupedProblem* probs, int count, void* ws, unsigned* status, uint64_t wait_ns,
                          int num_sms, cudaStream_t s) {
  if (count <= 0) return cudaSuccess;
  const DcPlan pl = dc_plan(probs, count, num_sms);
  static DcParams prm;  // 20+ KB: not on the host stack; launches copy it
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  prm.count = count;
  prm.grid = pl.grid;
  prm.maxseg = pl.maxseg;
  prm.units = pl.units;
  prm.slices = pl.slices;
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
    d.ypart = reinterpret_cast<float*>(base + pl.off_ypart[i]);
    d.cnt = reinterpret_cast<unsigned*>(base + pl.off_cnt[i]);
    d.n = static_cast<int>(g.w.n);
    d.k = static_cast<int>(g.w.k);
    d.m = g.m;
    d.r = g.r;
    d.scale = g.alpha / static_cast<float>(g.r);
    d.t_slices = pl.t_slices[i];
    d.t_w = pl.t_w[i];
    d.s0 = pl.s0[i];
    d.tiles = pl.tiles[i];
    d.ku = pl.ku[i];
    d.u0_w = pl.u0_w[i];
    if (g.m > mmax) mmax = g.m;
  }
  constexpr size_t kLut = 256 * 32 * 4;
  cudaError_t e0 = mmax <= 8 ? set_smem_limit_once(k_decode<1>, kLut) : set_smem_limit_once(k_decode<2>, kLut);
  if (e0 != cudaSuccess) return e0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kDcThreads);
  cfg.dynamicSmemBytes = kLut;
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
