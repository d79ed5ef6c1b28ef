// Grouped small-token forward (decode): Y_p = X_p deq(W_p)^T + s_p (X_p A_p^T) B_p^T
// for a list of independent problems p (1..16 tokens each), in two launches:
// k_lora_down_grouped, then one GEMV over every weight of the list --
//   k_gemv_cc_wide   CUDA cores, at most 2 tokens, lists with at least one
//                    128-row tile per CTA slot (a whole layer stack);
//   k_gemv_cc        CUDA cores, at most 4 tokens, shorter lists (one decoder
//                    layer's q,k,v or gate,up): 16-row tiles, k split over
//                    the SMs when the tiles do not fill them;
//   k_qgemv_grouped  tensor cores, everything else (up to 16 tokens).
//
// Glossary "QLoRA", "How QLoRA works": the frozen layer dequantises NF4 to
// bf16 before the matmul and adds the LoRA output; Day 25 notes section 4.4:
// inference runs the 4-bit base with the adapter attached.  With few tokens the
// step is a stream over the weight codes, so what matters is keeping HBM busy.
//
// k_lora_down_grouped  one CTA per problem: st_p = bf16(s_p X_p A_p^T) (and
//                      X_p A_p^T in f32 if asked), 16 warps splitting k; it
//                      lets the GEMV launch right after it has waited for its
//                      own predecessor, and the CUDA-core GEMVs wait for it
//                      only before their LoRA term.
// k_qgemv_grouped      work item = (problem, 128-row tile), dealt round-robin
//                      to the CTAs.  Per 64-wide k block ("stage"):
//   - a stage is two 64-wide k blocks; producer warps 1-4 decode the even
//     block, warps 5-8 the odd one, one weight row per thread, into TMEM
//     (tcgen05 A operand, M = 128): a weight pair is a bf16 (L[hi], L[lo])
//     pair from a byte-indexed shared-memory table (one column per lane, no
//     bank conflicts) times bf16(a') in one packed multiply (within a bf16
//     rounding of bf16(L a'); the fwd/bwd GEMMs keep the exact bf16(L a')).
//     Each thread prefetches its row's codes, block-scale byte, group step and
//     mean, plus one 16-byte slice of the 16-token activation tile (later of
//     the sT tile), with cp.async into a private shared-memory ring kPrefetch
//     stages ahead, with a meta word that tells the consuming pass what the
//     stage is; after the stage frees, the slice goes into the 128-byte
//     swizzled K-major B operand;
//   - one thread issues tcgen05.mma (N = 16) into a double-buffered TMEM
//     accumulator; the LoRA up-projection is the item's last stage(s);
//   - the producers drain item j's accumulator after producing item j+1.
// Deterministic: every output element is written once (the split CUDA-core
// path adds its float32 partial sums in a fixed order).
#include <cstdio>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace qlora {

constexpr int kGvMaxProbs = 300;

struct GvProb {
  const uint8_t* codes;
  const int8_t* absq;
  const float* step;
  const float* mean;
  const __nv_bfloat16* x;       // [m, k]
  const __nv_bfloat16* lora_b;  // [n, r]
  const __nv_bfloat16* st;      // [m, r]  bf16(s x A^T)
  __nv_bfloat16* y;             // [m, n]
  float* part;                  // [splits][m][n] float32 partial sums (CUDA-core path with splits > 1)
  unsigned* cnt;                // [row tiles] arrival counters of the splits (zeroed by the LoRA-down launch)
  int n, k, m, r;
  int item0;  // first work item of this problem
  int pad;
};

struct GvParams {
  int count, total_items;
  int splits;  // CUDA-core path: k splits per row tile
  int group;   // CUDA-core path: consecutive row tiles per work item
  unsigned long long wait_ns;
  unsigned* status;
  GvProb prob[kGvMaxProbs];
};

struct GlProb {
  const __nv_bfloat16* x;   // [m, k]
  const __nv_bfloat16* a;   // [r, k]
  __nv_bfloat16* st;        // [m, r]
  float* t_save;            // [m, r] or null
  int m, k, r;
  float scale;
};

struct GlParams {
  int count;
  int n_cnt;      // split counters to zero before the GEMV launch
  unsigned* cnt;
  GlProb prob[kGvMaxProbs];
};

__device__ __forceinline__ void mma_m16n8k16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ====================================================================== grouped LoRA down
// Same k-permuted m16n8k16 fragments as k_lora_down; one CTA per problem, 16
// warps over k, fixed-order reduction of the warps' partial sums.
template <int NT>
__global__ void __launch_bounds__(512) k_lora_down_grouped(const __grid_constant__ GlParams p) {
  constexpr int RP = NT * 8;
  // X may come from the kernel before, and that kernel may be the previous
  // call's GEMV still reading this workspace: wait for it, then let the GEMV
  // of this call start (it waits for this kernel before it needs sT)
  griddep_wait();
  griddep_launch_dependents();
  for (int i = blockIdx.x * 512 + threadIdx.x; i < p.n_cnt; i += gridDim.x * 512) p.cnt[i] = 0u;
  extern __shared__ float s_red_flat[];  // [16 warps][16 rows][RP]
  auto s_red = reinterpret_cast<float(*)[16 * RP]>(s_red_flat);
  const GlProb& pr = p.prob[blockIdx.x];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, q = lane & 3;
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  const int n_chunks = pr.k / 32;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  constexpr int U = NT <= 2 ? 4 : 2;
  for (int c = warp; c < n_chunks; c += 16 * U) {
    uint4 xa[U], xb[U], bv[U][NT];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cc = c + 16 * u;
      const int kb = cc * 32 + q * 8;
      const bool kin = cc < n_chunks;
      xa[u] = (kin && g < pr.m) ? ldg_nc_v4(pr.x + static_cast<int64_t>(g) * pr.k + kb) : zero;
      xb[u] = (kin && g + 8 < pr.m) ? ldg_nc_v4(pr.x + static_cast<int64_t>(g + 8) * pr.k + kb) : zero;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        const int j = t * 8 + g;
        bv[u][t] = (kin && j < pr.r) ? ldg_nc_v4(pr.a + static_cast<int64_t>(j) * pr.k + kb) : zero;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        mma_m16n8k16(acc[t], xa[u].x, xb[u].x, xa[u].y, xb[u].y, bv[u][t].x, bv[u][t].y);
        mma_m16n8k16(acc[t], xa[u].z, xb[u].z, xa[u].w, xb[u].w, bv[u][t].z, bv[u][t].w);
      }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int col = t * 8 + 2 * q;
    s_red[warp][g * RP + col] = acc[t][0];
    s_red[warp][g * RP + col + 1] = acc[t][1];
    s_red[warp][(g + 8) * RP + col] = acc[t][2];
    s_red[warp][(g + 8) * RP + col + 1] = acc[t][3];
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < 16 * RP; idx += 512) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 16; ++w) v += s_red[w][idx];
    const int row = idx / RP, j = idx % RP;
    if (row >= pr.m || j >= pr.r) continue;
    if (pr.t_save) pr.t_save[row * pr.r + j] = v;
    pr.st[row * pr.r + j] = __float2bfloat16_rn(__fmul_rn(v, pr.scale));
  }
}

// ====================================================================== grouped decode GEMV
constexpr int kGvThreads = 288;  // warp 0 MMA + TMEM, warps 1..8 producers
constexpr int kGvStages = 3;     // TMEM / smem ring depth (a stage = two 64-wide k blocks)
constexpr int kGvPrefetch = 4;   // producer cp.async distance, in stages
constexpr int kGvTok = 16;       // MMA N
constexpr uint32_t kGvBBytes = 2 * kGvTok * 128;  // two 64-wide slabs of 16 token rows
constexpr uint32_t kGvDCol = kGvStages * 64;
constexpr uint32_t kGvTmemCols = 256;
constexpr uint32_t kGvSlot = 64;
constexpr size_t kGvTab = 256 * 32 * 4;  // level-pair table, one column per lane
constexpr size_t kGvSmem =
    1024 + kGvStages * kGvBBytes + 256 * kGvPrefetch * kGvSlot + kGvTab + (2 * kGvStages + 4) * 8 + 16;
static_assert(kGvDCol + 2 * kGvTok <= kGvTmemCols, "TMEM budget");

// Slots of a prefetched stage, one per producer thread, stored field by field
// (structure of arrays: consecutive threads at consecutive 16- or 4-byte
// addresses, so the slot reads and the cp.async writes are free of bank
// conflicts): codes of the thread's row and k block (two 16-byte halves),
// activation slice, word holding the block-scale byte, group step, per-tensor
// mean, meta (written by the thread).
constexpr uint32_t kGvFCode0 = 0, kGvFCode1 = 16 * 256, kGvFAct = 32 * 256, kGvFScale = 48 * 256,
                   kGvFStep = 52 * 256, kGvFMean = 56 * 256, kGvFMeta = 60 * 256;
enum : uint32_t {
  kMetaValid = 1u,      // the stage exists
  kMetaLora = 2u,       // LoRA stage (A = B rows, B operand = sT)
  kMetaRowOk = 4u,      // row < n and the k block (or j block) is inside the matrix
  kMetaLast = 32u,      // last stage of its work item
};
// meta bits 3-4: byte of the scale word; bits 16-31: problem index

__device__ __forceinline__ int gv_find_prob(const GvParams& p, int item) {
  int lo = 0, hi = p.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.prob[mid].item0 <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Walks the stages of this CTA's work items (item = blockIdx.x + j * gridDim.x)
// with the current problem's fields cached in registers.
struct GvWalk {
  int j, l, nst, nmain, kb;  // item counter, stage in item, stages, main stages, k blocks
  int p, rt;
  bool done;
  const uint8_t* codes;
  const int8_t* absq;
  const float* step;
  const float* mean;
  const __nv_bfloat16* x;
  const __nv_bfloat16* st;
  int n, k, m, r;
};

__device__ __forceinline__ void gv_set_item(const GvParams& p, GvWalk& w) {
  const int item = blockIdx.x + w.j * gridDim.x;
  w.done = item >= p.total_items;
  if (w.done) return;
  w.p = gv_find_prob(p, item);
  const GvProb& pr = p.prob[w.p];
  w.rt = item - pr.item0;
  w.codes = pr.codes;
  w.absq = pr.absq;
  w.step = pr.step;
  w.mean = pr.mean;
  w.x = pr.x;
  w.st = pr.st;
  w.n = pr.n;
  w.k = pr.k;
  w.m = pr.m;
  w.r = pr.r;
  w.kb = pr.k / 64;
  w.nmain = (w.kb + 1) / 2;
  w.nst = w.nmain + 1;  // one LoRA stage: r <= 128 = two 64-wide j blocks
  w.l = 0;
}

__device__ __forceinline__ void gv_begin(const GvParams& p, GvWalk& w) {
  w.j = 0;
  gv_set_item(p, w);
}

__device__ __forceinline__ void gv_next(const GvParams& p, GvWalk& w) {
  if (++w.l >= w.nst) {
    ++w.j;
    gv_set_item(p, w);
  }
}

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* gptr) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(gptr) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t saddr, const void* gptr) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(saddr), "l"(gptr) : "memory");
}
__device__ __forceinline__ void cp_async16_zfill(uint32_t saddr, const void* gptr, bool valid) {
  const int src = valid ? 16 : 0;  // 0 source bytes: the 16 destination bytes are zero-filled
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(saddr), "l"(gptr), "r"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ uint4 lds_v4(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr));
  return v;
}
__device__ __forceinline__ uint32_t lds_u32(uint32_t saddr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr));
  return v;
}
__device__ __forceinline__ void sts_u32(uint32_t saddr, uint32_t v) {
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}

// Prefetch this thread's share of stage `w` into its slot of the prefetch stage
// at `sa` (thread t): half h takes k block 2l+h of row `row`, and activation
// slice (token tt/8, chunk tt%8) of slab h.  Always commits one cp.async group.
__device__ __forceinline__ void gv_prefetch(const GvWalk& w, int half, int rlocal, int tt, uint32_t sa, int t) {
  uint32_t meta = 0;
  if (!w.done) {
    meta = kMetaValid | (static_cast<uint32_t>(w.p) << 16) | (w.l == w.nst - 1 ? kMetaLast : 0u);
    const int tok = tt >> 3, ch = tt & 7;
    const int row = w.rt * 128 + rlocal;
    if (w.l < w.nmain) {
      const int blk = 2 * w.l + half;
      const bool kin = blk < w.kb;
      if (kin && row < w.n) {
        const uint8_t* cp = w.codes + static_cast<int64_t>(row) * (w.k / 2) + blk * 32;
        cp_async16(sa + kGvFCode0 + t * 16, cp);
        cp_async16(sa + kGvFCode1 + t * 16, cp + 16);
        const int64_t ai = static_cast<int64_t>(row) * w.kb + blk;
        cp_async4(sa + kGvFScale + t * 4, w.absq + (ai & ~int64_t(3)));
        cp_async4(sa + kGvFStep + t * 4, w.step + (ai >> 8));
        cp_async4(sa + kGvFMean + t * 4, w.mean);
        meta |= kMetaRowOk | (static_cast<uint32_t>(ai & 3) << 3);
      }
      const bool v = kin && tok < w.m;
      cp_async16_zfill(sa + kGvFAct + t * 16, w.x + (v ? static_cast<int64_t>(tok) * w.k + blk * 64 + ch * 8 : 0), v);
    } else {
      meta |= kMetaLora;
      const int jb = half * 64;
      if (row < w.n && jb < w.r) meta |= kMetaRowOk;
      const int col = jb + ch * 8;
      const bool v = tok < w.m && col < w.r;
      cp_async16_zfill(sa + kGvFAct + t * 16, w.st + (v ? static_cast<int64_t>(tok) * w.r + col : 0), v);
    }
  }
  sts_u32(sa + kGvFMeta + t * 4, meta);
  cp_async_commit();
}

__global__ void __launch_bounds__(kGvThreads, 2) k_qgemv_grouped(const __grid_constant__ GvParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sb = smem;                             // [kGvStages][2 slabs][16 rows][128 B]
  uint8_t* slots = smem + kGvStages * kGvBBytes;  // [kGvPrefetch][256 threads][kGvSlot]
  uint32_t* tab = reinterpret_cast<uint32_t*>(slots + 256 * kGvPrefetch * kGvSlot);  // [256 bytes][32 lanes]
  uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(tab) + kGvTab);
  uint64_t* empty = full + kGvStages;
  uint64_t* acc_full = empty + kGvStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  volatile int* vabort = abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGvStages; ++s) {
      mbar_init(&full[s], 256);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 256);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_holder, kGvTmemCols);
  }
  // level pairs (L[hi nibble], L[lo nibble]) as bf16, same in every column
  for (int i = threadIdx.x; i < 256 * 32; i += kGvThreads) {
    const int b = i >> 5;
    const __nv_bfloat16 lo = __float2bfloat16_rn(nf4_level(b >> 4)), hi = __float2bfloat16_rn(nf4_level(b & 15));
    tab[i] = static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(&lo)) |
             (static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(&hi)) << 16);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kGvTok, 0, 0);
      int j = 0, g = 0;
      while (blockIdx.x + j * gridDim.x < p.total_items) {
        const int pi = gv_find_prob(p, blockIdx.x + j * gridDim.x);
        const int nst = (p.prob[pi].k / 64 + 1) / 2 + 1;
        const int buf = j & 1;
        if (!mbar_wait(&acc_empty[buf], ((j >> 1) & 1) ^ 1, p.wait_ns, vabort)) {
          abort_cta(p.status, abort_flag);
          break;
        }
        bool ok = true;
        for (int l = 0; l < nst; ++l, ++g) {
          const int s = g % kGvStages;
          if (!mbar_wait(&full[s], (g / kGvStages) & 1, p.wait_ns, vabort)) {
            abort_cta(p.status, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b_addr = smem_u32(sb + s * kGvBBytes);
          const uint32_t d_tmem = tbase + kGvDCol + buf * kGvTok;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bdesc = sdesc_sw128(b_addr + (kk >> 2) * (kGvTok * 128) + (kk & 3) * 32, 16, 1024);
            mma_bf16_ts(d_tmem, tbase + s * 64 + kk * 8, bdesc, idesc, (l > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&acc_full[buf]);
        ++j;
      }
    }
  } else {
    // ------------------------------------------------------------ producers (+ deferred epilogue)
    const int half = (warp - 1) >> 2;              // k block 2l + half of each stage
    const int quarter = warp & 3;                  // TMEM lanes this warp may touch
    const int rlocal = quarter * 32 + lane;        // row within the 128-row tile
    const int t = threadIdx.x - 32;                // slot index 0..255
    const int tt = ((warp - 1) & 3) * 32 + lane;   // activation slice 0..127 of slab `half`
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t slot0 = smem_u32(slots);
    auto slot_addr = [&](int u) { return slot0 + static_cast<uint32_t>(u % kGvPrefetch) * 256 * kGvSlot; };

    GvWalk pre;
    gv_begin(p, pre);
    for (int u = 0; u < kGvPrefetch; ++u) {
      gv_prefetch(pre, half, rlocal, tt, slot_addr(u), t);
      if (!pre.done) gv_next(p, pre);
    }

    auto drain = [&](int jd) {
      const int buf = jd & 1;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (jd >> 1) & 1, p.wait_ns, vabort));
      ok = __all_sync(0xffffffffu, ok && !*vabort);
      if (ok) {
        tc_fence_after();
        const int item = blockIdx.x + jd * gridDim.x;
        const int pi = gv_find_prob(p, item);
        const GvProb& pr = p.prob[pi];
        const int row = (item - pr.item0) * 128 + rlocal;
        uint32_t v[16];
        __syncwarp();
        tmem_ld_32x32b_x16(tbase + lane_field + kGvDCol + buf * kGvTok, v);
        tmem_ld_wait();
        if (row < pr.n) {
          __nv_bfloat16* yrow = pr.y + row;
          const int m = pr.m, n = pr.n;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float val = __uint_as_float(half ? v[8 + i] : v[i]);
            const int tok = half * 8 + i;
            if (tok < m) yrow[static_cast<int64_t>(tok) * n] = __float2bfloat16_rn(val);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
      return ok;
    };

    int u = 0, j = 0;
    bool alive = true;
    while (alive) {
      cp_async_wait<kGvPrefetch - 1>();
      const uint32_t sa = slot_addr(u);
      const uint32_t meta = lds_u32(sa + kGvFMeta + t * 4);
      if (!(meta & kMetaValid)) break;
      const int s = u % kGvStages;
      const uint32_t ph = (u / kGvStages) & 1;
      const uint4 act = lds_v4(sa + kGvFAct + t * 16);
      uint32_t words[32];
      if (!(meta & kMetaRowOk)) {
#pragma unroll
        for (int c = 0; c < 32; ++c) words[c] = 0;
      } else if (!(meta & kMetaLora)) {
        const uint4 c0 = lds_v4(sa + kGvFCode0 + t * 16), c1 = lds_v4(sa + kGvFCode1 + t * 16);
        const uint32_t qw = lds_u32(sa + kGvFScale + t * 4);
        const int8_t qv = static_cast<int8_t>((qw >> (8 * ((meta >> 3) & 3))) & 0xffu);
        const float a2 = restore_absmax(qv, __uint_as_float(lds_u32(sa + kGvFStep + t * 4)),
                                        __uint_as_float(lds_u32(sa + kGvFMean + t * 4)));
        // weight pair = bf16(L) pair (one conflict-free table load) times bf16(a') in one packed multiply
        const __nv_bfloat162 a2b = __float2bfloat162_rn(a2);
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const uint32_t tab_me = smem_u32(tab) + lane * 4;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t e = lds_u32(tab_me + ((cw[i >> 2] >> (8 * (i & 3))) & 0xffu) * 128);
          const __nv_bfloat162 v = __hmul2(*reinterpret_cast<const __nv_bfloat162*>(&e), a2b);
          words[i] = *reinterpret_cast<const uint32_t*>(&v);
        }
      } else {
        const GvProb& pr = p.prob[meta >> 16];
        const int row = (blockIdx.x + j * gridDim.x - pr.item0) * 128 + rlocal;
        const uint32_t* brow = reinterpret_cast<const uint32_t*>(pr.lora_b + static_cast<int64_t>(row) * pr.r);
        const int jb = half * 64;
#pragma unroll
        for (int c = 0; c < 32; ++c) words[c] = (jb + 2 * c < pr.r) ? __ldg(brow + ((jb >> 1) + c)) : 0u;
      }
      // refill the slot with the stage kGvPrefetch ahead (its contents are in registers now)
      __syncwarp();
      gv_prefetch(pre, half, rlocal, tt, sa, t);
      if (!pre.done) gv_next(p, pre);

      const bool ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ph ^ 1, p.wait_ns, vabort));
      if (!ok) {
        if (lane == 0) abort_cta(p.status, abort_flag);
        alive = false;
        break;
      }
      tc_fence_after();
      sts_v4(smem_u32(sb + s * kGvBBytes) + half * (kGvTok * 128) + sw128_offset(tt >> 3, tt & 7), act.x, act.y,
             act.z, act.w);
      fence_proxy_async_smem();
      __syncwarp();
      tmem_st_32x32b_x32(tbase + lane_field + s * 64 + half * 32, words);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&full[s]);
      ++u;
      if (meta & kMetaLast) {
        // item j is fully produced: drain item j - 1 (its MMAs are done or nearly)
        if (j >= 1 && !drain(j - 1)) alive = false;
        ++j;
      }
    }
    if (alive && j >= 1) drain(j - 1);
    cp_async_wait<0>();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, kGvTmemCols);
  }
}

// ====================================================================== host
static_assert(sizeof(GvParams) <= 32000, "kernel parameter budget");
static_assert(sizeof(GlParams) <= 32000, "kernel parameter budget");

// ====================================================================== CUDA-core decode (1 or 2 tokens)
// With one or two tokens the tensor path is bound by its decode; here a weight
// pair costs a byte extract, one shared-memory load and two mixed-precision
// FMAs per token (fma.rn.f32.bf16: the bf16 x bf16 product is exact in
// float32, one rounding into the float32 sum).  The table holds, for every
// code byte, the bf16 pair (L[hi], L[lo]) with one column per lane (each lane
// reads its own bank); activations are staged as bf16, so the two halves of a
// staged word meet the two halves of a table word.  The block scale a'
// multiplies a 32-weight partial sum, so the level enters as bf16(L) times the
// float32 scale (the tensor path rounds bf16(L a'): both are within a bf16
// rounding of the exact product).
//
// Layout: a row tile is 16 rows, warp w owning rows 2 w and 2 w + 1; a k range
// is walked in segments of 1024 weights, lane l taking weights 32 l .. 32 l +
// 31 of each segment (half of a 64-block: one scale per lane and row), so
// every code load is 512 contiguous bytes of a row.  A work item is (problem,
// run of `group` consecutive tiles, k split): the item's activations (at most
// cc_max_k columns, the splits see to that) are staged once, 16 bytes of
// padding after every 32 columns so the lanes' chunks fall in different
// banks, and each warp walks the item's (tile, segment) pairs as one stream
// with the codes of the next kCcAhead pairs in registers.  The lanes' partial
// sums of a row meet in a warp reduction at the end of each tile.  When the
// tiles of a launch fill fewer than all CTA slots, each tile's k range is
// split: every split writes its float32 partial sums, and the last split to
// arrive (a per-tile counter) adds them in split order, adds the LoRA term and
// writes Y -- the result does not depend on the arrival order.
constexpr int kCcThreads = 256;
constexpr int kCcRowsPerWarp = 2;
constexpr int kCcRows = kCcRowsPerWarp * (kCcThreads / 32);  // rows per tile
constexpr int kCcCtasPerSm = 2;
constexpr int kCcSeg = 1024;    // weights per row per segment (32 lanes x 32)
constexpr int kCcAhead = 2;     // (tile, segment) pairs of codes in flight per warp beyond the current one
// staged activation columns of one item (two CTAs per SM at every token count)
__host__ __device__ constexpr int cc_max_k(int mt) { return mt <= 2 ? 12288 : 6144; }
__host__ __device__ constexpr int cc_xstride(int mt) { return cc_max_k(mt) / 32 * 40; }  // bf16 per staged token row (32 columns + 8 padding)
constexpr int kCcMaxSplits = 8;
template <int MT>
constexpr size_t cc_smem() {
  return 256 * 32 * 4 + static_cast<size_t>(MT) * cc_xstride(MT) * 2 + 16;
}

// acc += bf16(lo of x) * bf16(lo of l) + bf16(hi of x) * bf16(hi of l), each step rounded once in float32
__device__ __forceinline__ void cc_fma_pair(float& acc_lo, float& acc_hi, uint32_t x, uint32_t l) {
  asm("{\n\t.reg .b16 xl, xh, ll, lh;\n\t"
      "mov.b32 {xl, xh}, %2;\n\t"
      "mov.b32 {ll, lh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, xl, ll, %0;\n\t"
      "fma.rn.f32.bf16 %1, xh, lh, %1;\n\t}"
      : "+f"(acc_lo), "+f"(acc_hi)
      : "r"(x), "r"(l));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int MT>
__global__ void __launch_bounds__(kCcThreads, kCcCtasPerSm) k_gemv_cc(const __grid_constant__ GvParams p) {
  constexpr int R = kCcRowsPerWarp;
  constexpr int NS = kCcAhead + 1;  // register slots
  constexpr int kCcXStride = cc_xstride(MT);
  extern __shared__ __align__(16) uint32_t sm_cc[];
  uint32_t* tab = sm_cc;                                                  // [256 bytes][32 lanes]
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(sm_cc + 256 * 32);  // [MT][kCcXStride]
  int* s_last = reinterpret_cast<int*>(xs + MT * kCcXStride);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 256 * 32; i += kCcThreads) {
    const int b = i >> 5;  // byte: element 2i in the high nibble, 2i + 1 in the low nibble
    const __nv_bfloat16 lo = __float2bfloat16_rn(nf4_level(b >> 4)), hi = __float2bfloat16_rn(nf4_level(b & 15));
    tab[i] = static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(&lo)) |
             (static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(&hi)) << 16);
  }
  const uint32_t tab_me = smem_u32(tab) + lane * 4;
  const uint32_t xs_me = smem_u32(xs) + lane * 80;  // the lane's 32 columns of a segment
  const int S = p.splits, G = p.group;
  griddep_launch_dependents();  // the next launch waits for this grid before it touches anything of it
  for (int item = blockIdx.x; item < p.total_items; item += gridDim.x) {
    int lo_i = 0, hi_i = p.count - 1;  // problem of this item: last one with item0 <= item
    while (lo_i < hi_i) {
      const int mid = (lo_i + hi_i + 1) >> 1;
      if (p.prob[mid].item0 <= item) lo_i = mid; else hi_i = mid - 1;
    }
    const GvProb& pr = p.prob[lo_i];
    const int local = item - pr.item0, run = local / S, split = local - run * S;
    const int n = pr.n, k = pr.k, m = pr.m, r = pr.r;
    const int kb_row = k / 64;
    const int ntiles = (n + kCcRows - 1) / kCcRows;
    const int tile0 = run * G, tile_end = min(ntiles, tile0 + G);
    const int nseg = (k + kCcSeg - 1) / kCcSeg;
    const int per = (nseg + S - 1) / S;
    const int sg_begin = split * per, sg_end = min(nseg, sg_begin + per);
    const int nsg = sg_end > sg_begin ? sg_end - sg_begin : 0;
    const int npairs = (tile_end - tile0) * nsg;
    const float mu = *pr.mean;
    const int k_begin = sg_begin * kCcSeg, k_end = min(sg_end * kCcSeg, k);
    // codes and scale bytes of pair f = (tile tile0 + f / nsg, segment sg_begin + f % nsg), zero past the end
    // (the block's int8 scale and its group's step travel with the codes)
    auto load_pair = [&](int f, uint4 (&cw)[R], uint32_t (&qv)[R], float (&sv)[R]) {
      const bool in = f < npairs;
      const int tl = in ? tile0 + f / nsg : 0;
      const int kw = (in ? sg_begin + f % nsg : 0) * kCcSeg + lane * 32;
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int rw = tl * kCcRows + warp * R + q;
        const bool v = in && kw < k && rw < n;
        const int64_t blk = static_cast<int64_t>(rw) * kb_row + kw / 64;
        cw[q] = v ? ldg_nc_v4(pr.codes + static_cast<int64_t>(rw) * (k / 2) + kw / 2) : make_uint4(0, 0, 0, 0);
        qv[q] = v ? static_cast<uint32_t>(static_cast<uint8_t>(__ldg(pr.absq + blk))) : 0u;
        sv[q] = v ? __ldg(pr.step + (blk >> 8)) : 0.f;
      }
    };
    uint4 cw[NS][R];
    uint32_t qv[NS][R];
    float sq[NS][R];
#pragma unroll
    for (int d = 0; d < kCcAhead; ++d) load_pair(d, cw[d], qv[d], sq[d]);
    __syncthreads();  // the table is built; the previous item is done with xs
    // activations of the item's k range as bf16, 16-byte chunks (rows t >= m are zero)
    {
      const int len = k_end - k_begin;
      for (int i = tid; i < MT * (len / 8); i += kCcThreads) {
        const int t = i / (len / 8), k8 = (i - t * (len / 8)) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < m) v = __ldcg(reinterpret_cast<const uint4*>(pr.x + static_cast<int64_t>(t) * k + k_begin + k8));
        *reinterpret_cast<uint4*>(xs + t * kCcXStride + k8 + (k8 >> 5) * 8) = v;
      }
    }
    __syncthreads();
    float acc[R][MT];
    float bv[R][2];  // LoRA B entries of the tile's rows: lane j holds B[row][j] and B[row][j + 32]
    float sv[MT][2];  // sT of the item's problem, lanes over j (read once, after the wait below)
    bool have_st = false;
    int f = 0;
    for (int tl = tile0; tl < tile_end; ++tl) {
      int row[R];
      bool ok[R];
#pragma unroll
      for (int q = 0; q < R; ++q) {
        row[q] = tl * kCcRows + warp * R + q;
        ok[q] = row[q] < n;
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[q][t] = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = lane + 32 * h;
          bv[q][h] = (ok[q] && j < r) ? __bfloat162float(pr.lora_b[static_cast<int64_t>(row[q]) * r + j]) : 0.f;
        }
      }
      auto pair = [&](auto slot_c, int sg) {
        constexpr int cur = decltype(slot_c)::value;
        constexpr int nxt = (cur + kCcAhead) % NS;
        load_pair(f + kCcAhead, cw[nxt], qv[nxt], sq[nxt]);
        const int kw = sg * kCcSeg + lane * 32;
        const bool kin = kw < k;
        float a[R];  // block scales a' = q * step + mu of the lane's block in each row
#pragma unroll
        for (int q = 0; q < R; ++q)
          a[q] = (kin && ok[q]) ? restore_absmax(static_cast<int8_t>(qv[cur][q]), sq[cur][q], mu) : 0.f;
        float se[R][MT], so[R][MT];  // even / odd weight partial sums
#pragma unroll
        for (int q = 0; q < R; ++q)
#pragma unroll
          for (int t = 0; t < MT; ++t) se[q][t] = so[q][t] = 0.f;
        const uint32_t xk = xs_me + ((sg * kCcSeg - k_begin) / 32) * 80;
#pragma unroll
        for (int h = 0; h < 4; ++h) {  // 8 weights = one 32-bit code word per row
          uint4 xv[MT];
#pragma unroll
          for (int t = 0; t < MT; ++t) xv[t] = lds_v4(xk + t * (kCcXStride * 2) + h * 16);
#pragma unroll
          for (int q = 0; q < R; ++q) {
            const uint32_t cwd = h == 0 ? cw[cur][q].x : h == 1 ? cw[cur][q].y : h == 2 ? cw[cur][q].z : cw[cur][q].w;
#pragma unroll
            for (int bi = 0; bi < 4; ++bi) {
              uint32_t e;
              asm("ld.shared.u32 %0, [%1];" : "=r"(e) : "r"(tab_me + (prmt(cwd, 0u, 0x4440u | bi) << 7)));
#pragma unroll
              for (int t = 0; t < MT; ++t) {
                const uint32_t xw = bi == 0 ? xv[t].x : bi == 1 ? xv[t].y : bi == 2 ? xv[t].z : xv[t].w;
                cc_fma_pair(se[q][t], so[q][t], xw, e);
              }
            }
          }
        }
        if (kin) {  // past the last block the activations read are stale: nothing is added
#pragma unroll
          for (int q = 0; q < R; ++q)
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[q][t] = fmaf(a[q], se[q][t] + so[q][t], acc[q][t]);
        }
      };
      for (int sg = sg_begin; sg < sg_end; ++sg, ++f) {
        switch (f % NS) {  // the register slot of pair f (static inside each case)
          case 0: pair(std::integral_constant<int, 0>{}, sg); break;
          case 1: pair(std::integral_constant<int, 1>{}, sg); break;
          default: pair(std::integral_constant<int, 2>{}, sg); break;
        }
      }
#pragma unroll
      for (int q = 0; q < R; ++q)
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[q][t] = warp_sum(acc[q][t]);
      // sT and the zeroed split counters come from the LoRA-down launch before
      // this one; X did not (that launch waited for X's producer before it let
      // this grid start), so only this part waits for it
      griddep_wait();
      if (S > 1) {
        // this split's partial sums, then the last split of the tile finishes the rows
        if (lane == 0) {
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            if (t >= m) break;
            float* pp = pr.part + (static_cast<int64_t>(split) * m + t) * n;
#pragma unroll
            for (int q = 0; q < R; ++q)
              if (ok[q]) pp[row[q]] = acc[q][t];
          }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) *s_last = atomicAdd(pr.cnt + tl, 1u) == static_cast<unsigned>(S - 1);
        __syncthreads();
        const bool last = *s_last != 0;
        __syncthreads();  // every thread has read the flag before it is written for the next tile
        if (!last) continue;
        __threadfence();
        // lane q * MT + t adds the splits of row q, token t in split order
        float tot = 0.f;
        const int q_l = lane / MT, t_l = lane % MT;
        if (lane < R * MT && t_l < m) {
          int rr = n;
#pragma unroll
          for (int q = 0; q < R; ++q)
            if (q == q_l) rr = row[q];
          if (rr < n)
            for (int sp = 0; sp < S; ++sp) tot += __ldcg(pr.part + (static_cast<int64_t>(sp) * m + t_l) * n + rr);
        }
#pragma unroll
        for (int q = 0; q < R; ++q)
#pragma unroll
          for (int t = 0; t < MT; ++t) acc[q][t] = __shfl_sync(0xffffffffu, tot, q * MT + t);
      }
      // LoRA up-projection: + sum_j sT[t][j] B[row][j], lanes over j
      if (!have_st) {
        have_st = true;
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = lane + 32 * h;
            sv[t][h] = (t < m && j < r) ? __bfloat162float(__ldcg(pr.st + static_cast<int64_t>(t) * r + j)) : 0.f;
          }
      }
#pragma unroll
      for (int q = 0; q < R; ++q)
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const float l = warp_sum(fmaf(sv[t][0], bv[q][0], sv[t][1] * bv[q][1]));
          if (lane == 0 && t < m && ok[q])
            pr.y[static_cast<int64_t>(t) * n + row[q]] = __float2bfloat16_rn(acc[q][t] + l);
        }
    }
  }
}

// ---------------------------------------------------------------------- long lists
// When a list has at least one 128-row tile per CTA slot, per-item latency
// matters less than the steady stream, and this layout streams best: a work
// item is (problem, 128-row tile) over the whole k range; thread (g, c) of
// warp w owns rows 16 w + g and 16 w + g + 8 and the 32 contiguous weights c
// (0..3) of every 128-weight step; codes come through a per-thread cp.async
// ring (16 bytes per row per step) kCwDepth steps ahead, activations are
// staged as bf16 in windows of kCwWin columns (16 bytes of padding after every
// 32), the 4 lanes of a row are added with shuffles.  Same table, same
// mixed-precision FMAs and the same float32 block scale as k_gemv_cc.
constexpr int kCwRows = 128;
constexpr int kCwDepth = 8;
constexpr int kCwWin = 2048;
constexpr int kCwXStride = kCwWin / 32 * 40;  // bf16 per staged token row
template <int MT>
constexpr size_t cw_smem() {
  return 256 * 32 * 4 + static_cast<size_t>(kCwDepth) * kCcThreads * 32 + static_cast<size_t>(MT) * kCwXStride * 2;
}

template <int MT>
__global__ void __launch_bounds__(kCcThreads, kCcCtasPerSm) k_gemv_cc_wide(const __grid_constant__ GvParams p) {
  extern __shared__ __align__(16) uint32_t sm_cw[];
  uint32_t* tab = sm_cw;                                                      // [256 bytes][32 lanes]
  uint8_t* ring = reinterpret_cast<uint8_t*>(sm_cw + 256 * 32);               // [kCwDepth][2 rows][256 threads][16 B]
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(ring + kCwDepth * kCcThreads * 32);  // [MT][kCwXStride]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  for (int i = tid; i < 256 * 32; i += kCcThreads) {
    const int b = i >> 5;  // byte: element 2i in the high nibble, 2i + 1 in the low nibble
    const __nv_bfloat16 lo = __float2bfloat16_rn(nf4_level(b >> 4)), hi = __float2bfloat16_rn(nf4_level(b & 15));
    tab[i] = static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(&lo)) |
             (static_cast<uint32_t>(*reinterpret_cast<const unsigned short*>(&hi)) << 16);
  }
  const uint32_t ring_me = smem_u32(ring) + tid * 16;
  const uint32_t tab_me = smem_u32(tab) + lane * 4;
  const uint32_t xs_me = smem_u32(xs) + c * 80;  // the thread's 32 columns of a 128-column step
  griddep_launch_dependents();  // the next launch waits for this grid before it touches anything of it
  for (int item = blockIdx.x; item < p.total_items; item += gridDim.x) {
    int lo_i = 0, hi_i = p.count - 1;  // problem of this item: last one with item0 <= item
    while (lo_i < hi_i) {
      const int mid = (lo_i + hi_i + 1) >> 1;
      if (p.prob[mid].item0 <= item) lo_i = mid; else hi_i = mid - 1;
    }
    const GvProb& pr = p.prob[lo_i];
    const int n = pr.n, k = pr.k, m = pr.m, r = pr.r;
    const int row0 = (item - pr.item0) * kCwRows + warp * 16 + g, row1 = row0 + 8;
    const bool ok0 = row0 < n, ok1 = row1 < n;
    const int kb_row = k / 64, nsteps = (kb_row + 1) / 2;
    const float mu = *pr.mean;
    const uint8_t* cp0 = pr.codes + static_cast<int64_t>(ok0 ? row0 : 0) * (k / 2) + c * 16;
    const uint8_t* cp1 = pr.codes + static_cast<int64_t>(ok1 ? row1 : 0) * (k / 2) + c * 16;
    const int64_t ab0 = static_cast<int64_t>(ok0 ? row0 : 0) * kb_row, ab1 = static_cast<int64_t>(ok1 ? row1 : 0) * kb_row;
    auto issue = [&](int st) {  // step st's 32 weights of both rows into the ring
      const int kb = 2 * st + (c >> 1);
      if (st < nsteps && kb < kb_row) {
        const uint32_t slot = ring_me + (st % kCwDepth) * (kCcThreads * 32);
        if (ok0) cp_async16(slot, cp0 + st * 64);
        if (ok1) cp_async16(slot + kCcThreads * 16, cp1 + st * 64);
      }
      cp_async_commit();
    };
#pragma unroll 1
    for (int d = 0; d < kCwDepth - 1; ++d) issue(d);
    // the LoRA B entries of the two rows this thread adds at the end (r / 4 of each row, r <= 64)
    const int jq = r / 4;  // r % 8 == 0: even, so 4-byte loads are aligned
    uint32_t bw0[8], bw1[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool in = 2 * u < jq;
      bw0[u] = (ok0 && in) ? *reinterpret_cast<const uint32_t*>(pr.lora_b + static_cast<int64_t>(row0) * r + c * jq + 2 * u) : 0u;
      bw1[u] = (ok1 && in) ? *reinterpret_cast<const uint32_t*>(pr.lora_b + static_cast<int64_t>(row1) * r + c * jq + 2 * u) : 0u;
    }
    float acc0[MT], acc1[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc0[t] = acc1[t] = 0.f;
    uint32_t q4_0 = 0, q4_1 = 0;  // block-scale bytes of blocks 4 qb .. 4 qb + 3 (little-endian)
    int qb = -1;
    int g0 = -1, g1 = -1;         // double-quant groups of the cached steps
    float st0 = 0.f, st1 = 0.f;
    __syncthreads();  // the table is built; the previous item is done with xs
    for (int w0 = 0; w0 < k; w0 += kCwWin) {
      const int wlen = min(kCwWin, k - w0);
      for (int i = tid; i < MT * (wlen / 8); i += kCcThreads) {
        const int t = i / (wlen / 8), k8 = (i - t * (wlen / 8)) * 8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < m) v = __ldcg(reinterpret_cast<const uint4*>(pr.x + static_cast<int64_t>(t) * k + w0 + k8));
        *reinterpret_cast<uint4*>(xs + t * kCwXStride + k8 + (k8 >> 5) * 8) = v;
      }
      __syncthreads();
      const int s0 = w0 / 128, s1 = (w0 + wlen + 127) / 128;
      for (int st = s0; st < s1; ++st) {
        issue(st + kCwDepth - 1);
        const int kb = 2 * st + (c >> 1);
        const bool kin = kb < kb_row;
        if (kin && (kb >> 2) != qb) {  // 4 scale bytes at a time (kb_row % 4 == 0 keeps them aligned)
          qb = kb >> 2;
          const int kb4 = kb & ~3;
          if ((kb_row & 3) == 0) {
            if (ok0) q4_0 = *reinterpret_cast<const uint32_t*>(pr.absq + ab0 + kb4);
            if (ok1) q4_1 = *reinterpret_cast<const uint32_t*>(pr.absq + ab1 + kb4);
          } else {
            q4_0 = q4_1 = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              if (kb4 + e < kb_row) {
                if (ok0) q4_0 |= static_cast<uint32_t>(static_cast<uint8_t>(pr.absq[ab0 + kb4 + e])) << (8 * e);
                if (ok1) q4_1 |= static_cast<uint32_t>(static_cast<uint8_t>(pr.absq[ab1 + kb4 + e])) << (8 * e);
              }
            }
          }
        }
        const int gr0 = static_cast<int>((ab0 + kb) >> 8), gr1 = static_cast<int>((ab1 + kb) >> 8);
        if (kin && gr0 != g0) { g0 = gr0; st0 = ok0 ? pr.step[gr0] : 0.f; }
        if (kin && gr1 != g1) { g1 = gr1; st1 = ok1 ? pr.step[gr1] : 0.f; }
        const int sh = 8 * (kb & 3);
        const float a0 = (ok0 && kin) ? restore_absmax(static_cast<int8_t>((q4_0 >> sh) & 0xffu), st0, mu) : 0.f;
        const float a1 = (ok1 && kin) ? restore_absmax(static_cast<int8_t>((q4_1 >> sh) & 0xffu), st1, mu) : 0.f;
        cp_async_wait<kCwDepth - 1>();
        const uint32_t slot = ring_me + (st % kCwDepth) * (kCcThreads * 32);
        const uint4 cw0 = lds_v4(slot), cw1 = lds_v4(slot + kCcThreads * 16);
        const uint32_t wr0[4] = {cw0.x, cw0.y, cw0.z, cw0.w}, wr1[4] = {cw1.x, cw1.y, cw1.z, cw1.w};
        float s0e[MT], s0o[MT], s1e[MT], s1o[MT];  // even / odd weight partial sums of the two rows
#pragma unroll
        for (int t = 0; t < MT; ++t) s0e[t] = s0o[t] = s1e[t] = s1o[t] = 0.f;
        const uint32_t xk = xs_me + ((st * 128 - w0) / 128) * 320;  // 4 chunks of 80 bytes per step
#pragma unroll
        for (int h = 0; h < 4; ++h) {  // 8 weights = one 32-bit code word per row
          uint4 xv[MT];
#pragma unroll
          for (int t = 0; t < MT; ++t) xv[t] = lds_v4(xk + t * (kCwXStride * 2) + h * 16);
          const uint32_t c0w = (ok0 && kin) ? wr0[h] : 0u, c1w = (ok1 && kin) ? wr1[h] : 0u;
#pragma unroll
          for (int bi = 0; bi < 4; ++bi) {
            uint32_t e0, e1;
            asm("ld.shared.u32 %0, [%1];" : "=r"(e0) : "r"(tab_me + (prmt(c0w, 0u, 0x4440u | bi) << 7)));
            asm("ld.shared.u32 %0, [%1];" : "=r"(e1) : "r"(tab_me + (prmt(c1w, 0u, 0x4440u | bi) << 7)));
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              const uint32_t xw = bi == 0 ? xv[t].x : bi == 1 ? xv[t].y : bi == 2 ? xv[t].z : xv[t].w;
              cc_fma_pair(s0e[t], s0o[t], xw, e0);
              cc_fma_pair(s1e[t], s1o[t], xw, e1);
            }
          }
        }
        if (kin) {  // past the last block the activations read are stale: nothing is added
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            acc0[t] = fmaf(a0, s0e[t] + s0o[t], acc0[t]);
            acc1[t] = fmaf(a1, s1e[t] + s1o[t], acc1[t]);
          }
        }
      }
      __syncthreads();  // xs is rewritten by the next window
    }
    cp_async_wait<0>();
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      acc0[t] += __shfl_xor_sync(0xffffffffu, acc0[t], 1);
      acc0[t] += __shfl_xor_sync(0xffffffffu, acc0[t], 2);
      acc1[t] += __shfl_xor_sync(0xffffffffu, acc1[t], 1);
      acc1[t] += __shfl_xor_sync(0xffffffffu, acc1[t], 2);
    }
    griddep_wait();  // sT comes from the LoRA-down launch before this one
    // LoRA up-projection: + sum_j st[t][j] B[row][j]; the 4 lanes of a row split j
    float l0[MT], l1[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) l0[t] = l1[t] = 0.f;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      if (jj < jq) {
        const int j = c * jq + jj;
        const float b0 = __uint_as_float((jj & 1) ? (bw0[jj >> 1] & 0xffff0000u) : (bw0[jj >> 1] << 16));
        const float b1 = __uint_as_float((jj & 1) ? (bw1[jj >> 1] & 0xffff0000u) : (bw1[jj >> 1] << 16));
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const float sv = t < m ? __bfloat162float(__ldcg(pr.st + static_cast<int64_t>(t) * r + j)) : 0.f;
          l0[t] = fmaf(sv, b0, l0[t]);
          l1[t] = fmaf(sv, b1, l1[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      l0[t] += __shfl_xor_sync(0xffffffffu, l0[t], 1);
      l0[t] += __shfl_xor_sync(0xffffffffu, l0[t], 2);
      l1[t] += __shfl_xor_sync(0xffffffffu, l1[t], 1);
      l1[t] += __shfl_xor_sync(0xffffffffu, l1[t], 2);
    }
    if (c == 0) {
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        if (t >= m) break;
        if (ok0) pr.y[static_cast<int64_t>(t) * n + row0] = __float2bfloat16_rn(acc0[t] + l0[t]);
        if (ok1) pr.y[static_cast<int64_t>(t) * n + row1] = __float2bfloat16_rn(acc1[t] + l1[t]);
      }
    }
  }
}

int fwd_grouped_max_problems() { return kGvMaxProbs; }

// Work plan of one launch: which GEMV, the k splits of the CUDA-core path,
// and the workspace regions (bf16 sT per problem, float32 partials, tile
// counters), each 256-byte aligned.
struct GroupedPlan {
  bool cuda_core;
  bool wide;  // CUDA-core path, long list: k_gemv_cc_wide
  int mmax, rmax, splits, group, items;
  size_t st_bytes, part_bytes, cnt_bytes;
};

static size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Launch with programmatic stream serialisation: the kernel may start while the
// one before it in the stream finishes; it waits (griddepcontrol.wait) before
// it reads anything that kernel writes.
template <typename P>
static cudaError_t launch_dependent(void (*kernel)(P), int grid, int block, size_t smem, cudaStream_t s, const P& prm) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, prm);
}

static GroupedPlan plan_grouped(const GroupedProblem* probs, int count, int num_sms) {
  GroupedPlan pl = {};
  pl.mmax = 1;
  pl.rmax = 8;
  int tiles = 0, nsteps_min = 1 << 30;
  for (int i = 0; i < count; ++i) {
    if (probs[i].m > pl.mmax) pl.mmax = probs[i].m;
    if (probs[i].r > pl.rmax) pl.rmax = probs[i].r;
    tiles += static_cast<int>((probs[i].w.n + kCcRows - 1) / kCcRows);
    const int nseg = static_cast<int>((probs[i].w.k + kCcSeg - 1) / kCcSeg);
    if (nseg < nsteps_min) nsteps_min = nseg;
    pl.st_bytes += align256(static_cast<size_t>(probs[i].m) * probs[i].r * 2);
  }
  pl.cuda_core = pl.mmax <= 2;
  pl.splits = 1;
  pl.group = 1;
  int tiles_wide = 0;
  for (int i = 0; i < count; ++i) tiles_wide += static_cast<int>((probs[i].w.n + kCwRows - 1) / kCwRows);
  pl.wide = pl.cuda_core && tiles_wide >= kCcCtasPerSm * num_sms;
  // short lists of 3 or 4 tokens take the split CUDA-core layout as well (the
  // tensor path's 128-row tiles would leave most SMs idle)
  if (!pl.cuda_core && pl.mmax <= 4 && tiles_wide < kCcCtasPerSm * num_sms) pl.cuda_core = true;
  if (pl.wide) {
    pl.items = tiles_wide;
  } else if (pl.cuda_core) {
    // every split's k range fits the staged activations; more splits when the
    // tiles leave CTA slots idle (at least 2 segments per split)
    const int slots = kCcCtasPerSm * num_sms;
    int kmax = 64;
    for (int i = 0; i < count; ++i)
      if (probs[i].w.k > kmax) kmax = static_cast<int>(probs[i].w.k);
    const int s_min = (kmax + cc_max_k(pl.mmax) - 1) / cc_max_k(pl.mmax);
    int s = 1;
    if (tiles > 0 && tiles < slots) s = slots / tiles;
    if (s > kCcMaxSplits) s = kCcMaxSplits;
    if (s > nsteps_min / 2) s = nsteps_min / 2;
    pl.splits = s > s_min ? s : s_min;
    // runs of consecutive tiles per item: about 4 items per CTA slot
    const long long work = static_cast<long long>(tiles) * pl.splits;
    if (work > 4LL * slots) pl.group = static_cast<int>(work / (4LL * slots));
    pl.items = 0;
    for (int i = 0; i < count; ++i) {
      const int t = static_cast<int>((probs[i].w.n + kCcRows - 1) / kCcRows);
      pl.items += (t + pl.group - 1) / pl.group * pl.splits;
    }
    if (pl.splits > 1) {
      for (int i = 0; i < count; ++i)
        pl.part_bytes += align256(static_cast<size_t>(pl.splits) * probs[i].m * probs[i].w.n * 4);
      pl.cnt_bytes = align256(static_cast<size_t>(tiles) * 4);
    }
  } else {
    pl.items = 0;
    for (int i = 0; i < count; ++i) pl.items += static_cast<int>((probs[i].w.n + 127) / 128);
  }
  return pl;
}

size_t fwd_grouped_workspace_bytes(const GroupedProblem* probs, int count, int num_sms) {
  const GroupedPlan pl = plan_grouped(probs, count, num_sms);
  return pl.st_bytes + pl.part_bytes + pl.cnt_bytes;
}

cudaError_t launch_fwd_grouped(const GroupedProblem* probs, int count, void* ws, unsigned* status, uint64_t wait_ns,
                               int num_sms, cudaStream_t s) {
  static GvParams gv;  // host staging of the by-value parameter block (not thread safe by design: one caller)
  static GlParams gl;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  memset(&gv, 0, sizeof(gv));
  memset(&gl, 0, sizeof(gl));
  const GroupedPlan pl = plan_grouped(probs, count, num_sms);
  char* base = static_cast<char*>(ws);
  size_t off = 0, off_part = pl.st_bytes, off_cnt = pl.st_bytes + pl.part_bytes;
  int items = 0, tiles = 0;
  for (int i = 0; i < count; ++i) {
    const GroupedProblem& q = probs[i];
    __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(base + off);
    off += align256(static_cast<size_t>(q.m) * q.r * 2);
    GvProb& g = gv.prob[i];
    g.codes = q.w.codes;
    g.absq = q.w.absq;
    g.step = q.w.step;
    g.mean = q.w.mean;
    g.x = q.x;
    g.lora_b = q.lora_b;
    g.st = st;
    g.y = q.y;
    g.n = static_cast<int>(q.w.n);
    g.k = static_cast<int>(q.w.k);
    g.m = q.m;
    g.r = q.r;
    g.item0 = items;
    if (pl.wide) {
      items += (g.n + kCwRows - 1) / kCwRows;
    } else if (pl.cuda_core) {
      const int t = (g.n + kCcRows - 1) / kCcRows;
      items += (t + pl.group - 1) / pl.group * pl.splits;
      if (pl.splits > 1) {
        g.part = reinterpret_cast<float*>(base + off_part);
        off_part += align256(static_cast<size_t>(pl.splits) * q.m * g.n * 4);
        g.cnt = reinterpret_cast<unsigned*>(base + off_cnt) + tiles;
      }
      tiles += t;
    } else {
      items += (g.n + 127) / 128;
    }
    GlProb& l = gl.prob[i];
    l.x = q.x;
    l.a = q.lora_a;
    l.st = st;
    l.t_save = q.t_save;
    l.m = q.m;
    l.k = g.k;
    l.r = q.r;
    l.scale = q.alpha / static_cast<float>(q.r);
  }
  gv.count = count;
  gv.total_items = items;
  gv.splits = pl.splits;
  gv.group = pl.group;
  gv.wait_ns = wait_ns;
  gv.status = status;
  gl.count = count;
  if (pl.cuda_core && pl.splits > 1) {  // the LoRA-down launch zeroes the split counters
    gl.n_cnt = tiles;
    gl.cnt = reinterpret_cast<unsigned*>(base + off_cnt);
  }
  cudaError_t e;
  if (pl.rmax <= 16) {
    e = set_smem_limit_once(k_lora_down_grouped<2>, 16 * 16 * 16 * 4);
    if (e == cudaSuccess) e = launch_dependent(k_lora_down_grouped<2>, count, 512, 16 * 16 * 16 * 4, s, gl);
  } else if (pl.rmax <= 32) {
    e = set_smem_limit_once(k_lora_down_grouped<4>, 16 * 16 * 32 * 4);
    if (e == cudaSuccess) e = launch_dependent(k_lora_down_grouped<4>, count, 512, 16 * 16 * 32 * 4, s, gl);
  } else {
    e = set_smem_limit_once(k_lora_down_grouped<8>, 16 * 16 * 64 * 4);
    if (e == cudaSuccess) e = launch_dependent(k_lora_down_grouped<8>, count, 512, 16 * 16 * 64 * 4, s, gl);
  }
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (pl.cuda_core) {
    // CUDA-core decode for 1 or 2 token columns (with more, the FMAs per weight
    // catch up with the tensor path's decode cost)
    const int grid = items < kCcCtasPerSm * num_sms ? items : kCcCtasPerSm * num_sms;
#define QLORA_CC(MT)                                                                                       \
  do {                                                                                                     \
    if (pl.wide) {                                                                                         \
      e = set_smem_limit_once(k_gemv_cc_wide<MT>, cw_smem<MT>());                                          \
      if (e == cudaSuccess) e = launch_dependent(k_gemv_cc_wide<MT>, grid, kCcThreads, cw_smem<MT>(), s, gv); \
    } else {                                                                                               \
      e = set_smem_limit_once(k_gemv_cc<MT>, cc_smem<MT>());                                               \
      if (e == cudaSuccess) e = launch_dependent(k_gemv_cc<MT>, grid, kCcThreads, cc_smem<MT>(), s, gv);   \
    }                                                                                                      \
  } while (0)
    if (pl.mmax == 1) {
      QLORA_CC(1);
    } else if (pl.mmax == 2) {
      QLORA_CC(2);
    } else {  // 3 or 4 tokens, short list (never the long-list layout)
      e = set_smem_limit_once(k_gemv_cc<4>, cc_smem<4>());
      if (e == cudaSuccess) e = launch_dependent(k_gemv_cc<4>, grid, kCcThreads, cc_smem<4>(), s, gv);
    }
#undef QLORA_CC
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  int grid = 2 * num_sms;
  if (grid > items) grid = items;
  e = set_smem_limit_once(k_qgemv_grouped, kGvSmem);
  if (e != cudaSuccess) return e;
  k_qgemv_grouped<<<grid, kGvThreads, kGvSmem, s>>>(gv);
  return cudaGetLastError();
}

}  // namespace qlora
