// tcgen05 GEMMs of the QLoRA NF4 linear.
//
// Glossary "QLoRA", "How QLoRA works": every frozen layer dequantises its NF4
// weight to bfloat16 before the matmul and adds the LoRA output; gradients
// flow through the dequantised weight into the two LoRA matrices only.  Day 25
// notes, sections 2.1 / 6.2: output W0 x + s B A x with s = alpha / r.
//
// Here the dequantised weight never reaches HBM: producer warps decode NF4
// codes straight into tensor-core operands.
//
// k_qgemm_wa  (forward and small-token decode)
//   D^T[n, m] = sum_k deq(W)[n, k] X[m, k]  +  sum_j B[n, j] sT[m, j]
//   A operand = 128 rows of deq(W) (then of LoRA B), written by the producers
//               into TMEM with tcgen05.st (one thread = one row = one TMEM lane,
//               one 64-wide k block = one absmax block = 32 TMEM columns);
//   B operand = NTOK token rows of X (then of sT = bf16(s X A^T)), TMA, 128B swizzle.
//   The LoRA up-projection is one (or two, r > 64) extra k blocks of the same
//   accumulator.  Few tiles: k split over the CTAs of a cluster, whose results
//   are added in split order through distributed shared memory.
// k_qgemm_wb  (backward dX)
//   D[m, k] = sum_n dY[m, n] deq(W)[n, k]  +  sum_j sU[m, j] A[j, k]
//   A operand = 2 x 128 token rows of dY (then sU = bf16(s dY B)), TMA, two
//               accumulators sharing each dequantised B block;
//   B operand = deq(W)[n-block of 64, 256 output columns], MN-major 128B swizzle,
//               written by the producers with st.shared (then LoRA A rows, TMA).
//   Few tiles: n split over the CTAs of a cluster, added as in k_qgemm_wa.
// k_lora_grad (LoRA gradients, both MN-major operands, HBM-bound)
//   dA^T[k, j] = sum_m X[m, k] sU[m, j],   dB[n, j] = sum_m dY[m, n] sT[m, j].
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "kernels.h"

namespace qlora {


// ====================================================================== forward / decode
struct WaParams {
  const uint8_t* codes;
  const int8_t* absq;
  const float* step;
  const float* mean;
  const __nv_bfloat16* lora_b;  // [N, r]
  __nv_bfloat16* y;             // [M, N]
  unsigned* status;
  int M, N, K, r;
  int kb_per_split, splits, lora_blocks;  // k split over `splits` CTAs of one cluster (the last adds LoRA)
  unsigned long long wait_ns;
};

constexpr int kWaTeams = 4;      // producer teams (4 warps each) taking k blocks round-robin
// split ways of the small-token GEMMs: clusters of up to 4 CTAs (one per SM); clusters of 8
// measured slower -- they need 8 free SMs of one GPC at once beside the other kernels
constexpr int kMaxSplitK = 4;

// 16-byte store into the shared memory of CTA `rank` of the cluster, at the offset `local` has here.
__device__ __forceinline__ void st_cluster_v4(uint32_t local, uint32_t rank, float4 v) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(local), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(ra), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}
constexpr int kWaThreads = 64 + kWaTeams * 128;  // warp 0: TMA + TMEM alloc, warp 1: MMA, then the producer teams

template <int NTOK, int STAGES>
struct WaCfg {
  static constexpr uint32_t kBBytes = NTOK * 128;
  static constexpr uint32_t kDCol = STAGES * 32;
  static constexpr uint32_t kTmemCols =
      (kDCol + NTOK) <= 32 ? 32 : (kDCol + NTOK) <= 64 ? 64 : (kDCol + NTOK) <= 128 ? 128 : (kDCol + NTOK) <= 256 ? 256 : 512;
  static constexpr size_t kSmem = 1024 + STAGES * kBBytes + (2 * STAGES + 1) * 8 + 16;
  static_assert(kDCol + NTOK <= 512, "TMEM budget");
  static_assert(NTOK % 16 == 0 && NTOK >= 16 && NTOK <= 256, "MMA N for M = 128");
};

// The token columns a producer team reads back from the accumulator: NTOK / 4 each, or all of
// them for team 0 when that share would be under 16 (one 16-column TMEM load).
template <int NTOK>
__device__ __forceinline__ int wa_col_lo(int team) {
  return (NTOK / kWaTeams) >= 16 ? team * (NTOK / kWaTeams) : 0;
}
template <int NTOK>
__device__ __forceinline__ int wa_ncols(int team) {
  return (NTOK / kWaTeams) >= 16 ? NTOK / kWaTeams : (team == 0 ? NTOK : 0);
}

template <int NTOK, int STAGES>
__global__ void __launch_bounds__(kWaThreads, 1)
    k_qgemm_wa(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_st, const WaParams p) {
  using Cfg = WaCfg<NTOK, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sb = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::kBBytes);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  volatile int* vabort = abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // split = this CTA's rank in its cluster (clusters of `splits` CTAs along z)
  const int n0 = blockIdx.x * 128, tok0 = blockIdx.y * NTOK, split = blockIdx.z;
  const int kb_total = p.K / 64;
  const int kb_begin = split * p.kb_per_split;
  const int kb_end = min(kb_total, kb_begin + p.kb_per_split);
  const int n_main = kb_end - kb_begin;
  const int n_iter = n_main + (split == p.splits - 1 ? p.lora_blocks : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1 + 128);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;
  bool prod_ok = false;  // producers: the accumulator holds this CTA's result

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_st);
      for (int i = 0; i < n_iter; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); break; }
        if (i == n_main) griddep_wait();  // sT is written by the preceding LoRA down kernel
        mbar_arrive_expect_tx(&full[s], Cfg::kBBytes);
        if (i < n_main)
          tma_load_2d(sb + s * Cfg::kBBytes, &tm_x, &full[s], (kb_begin + i) * 64, tok0);
        else
          tma_load_2d(sb + s * Cfg::kBBytes, &tm_st, &full[s], (i - n_main) * 64, tok0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, NTOK, 0, 0);
      const uint32_t d_tmem = tbase + Cfg::kDCol;
      for (int i = 0; i < n_iter; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&full[s], ph, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); break; }
        tc_fence_after();
        const uint32_t b_addr = smem_u32(sb + s * Cfg::kBBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bdesc = sdesc_sw128(b_addr + kk * 32, 16, 1024);
          mma_bf16_ts(d_tmem, tbase + s * 32 + kk * 8, bdesc, idesc, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(acc_full);
    }
  } else {
    // ---------------------------------------------------------------- producers
    const int team = (warp - 2) >> 2;
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 are the only ones this warp may touch
    const int row = n0 + quarter * 32 + lane;
    const bool row_ok = row < p.N;
    const float mu = *p.mean;
    const int kb_row = p.K / 64;
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    // the codes and absmax of a k block are loaded one trip ahead of its decode
    const uint8_t* row_codes = p.codes + static_cast<int64_t>(row) * (p.K / 2);
    const int64_t row_abs = static_cast<int64_t>(row) * kb_row;
    uint4 nc0 = make_uint4(0, 0, 0, 0), nc1 = nc0;
    int8_t nq = 0;
    float nstep = 0.f;
    auto fetch = [&](int i) {
      if (i < n_main && row_ok) {
        const int kb = kb_begin + i;
        nc0 = ldg_nc_v4(row_codes + kb * 32);
        nc1 = ldg_nc_v4(row_codes + kb * 32 + 16);
        nq = p.absq[row_abs + kb];
        nstep = p.step[(row_abs + kb) >> 8];
      }
    };
    fetch(team);
    bool alive = true;
    for (int i = team; i < n_iter && alive; i += kWaTeams) {
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      uint32_t words[32];
      if (i < n_main) {
        const uint4 c0 = nc0, c1 = nc1;
        const float a2 = restore_absmax(nq, nstep, mu);
        fetch(i + kWaTeams);
        if (row_ok) {
          nf4_decode_block(c0, c1, a2, words);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) words[c] = 0;
        }
      } else {
        load_lora_b_row(p.lora_b, row, p.N, p.r, (i - n_main) * 64, words);
      }
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ph ^ 1, p.wait_ns, vabort));
      if (!ok) { if (lane == 0) abort_cta(p.status, abort_flag); alive = false; break; }
      tc_fence_after();
      __syncwarp();
      tmem_st_32x32b_x32(tbase + lane_field + s * 32, words);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&full[s]);
    }
    // ---------------------------------------------------------------- epilogue
    bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, p.wait_ns, vabort));
    ok = ok && !*vabort;
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    prod_ok = ok;
    if (ok && p.splits == 1) {
      const uint32_t dcol = tbase + lane_field + Cfg::kDCol;
      const int ncv = min(NTOK, p.M - tok0);  // columns that hold tokens
      for (int c = wa_col_lo<NTOK>(team); c < wa_col_lo<NTOK>(team) + wa_ncols<NTOK>(team) && c < ncv; c += 16) {
        uint32_t v[16];
        __syncwarp();
        tmem_ld_32x32b_x16(dcol + c, v);
        tmem_ld_wait();
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int tok = tok0 + c + j;
            if (tok < p.M) p.y[static_cast<int64_t>(tok) * p.N + row] = __float2bfloat16_rn(__uint_as_float(v[j]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (p.splits > 1) {
    // Split k: the accumulator's four TMEM lane quarters (32 weight rows each) are owned
    // round-robin (quarter q by the CTA of cluster rank q % splits).  Each CTA sends the quarters
    // it does not own, as float32 [token / 4][32 rows] float4 slices, into the owner's now idle
    // stage buffers -- slot s (s - 1 past the owner) for sender s, laid out [owned quarter
    // q / splits][token / 4][32 rows] -- and each owner adds the splits in split order and writes Y.
    tc_fence_after();
    cluster_sync();  // every CTA of the cluster is past its k loop: the stage buffers are free
    const int ncv = min(NTOK, p.M - tok0);
    const int team = (warp - 2) >> 2, quarter = warp & 3;
    const int o = quarter % p.splits;
    const uint32_t dcol = tbase + (static_cast<uint32_t>(quarter * 32) << 16) + Cfg::kDCol;
    const uint32_t base = smem_u32(smem);
    const uint32_t slot_bytes = static_cast<uint32_t>((4 + p.splits - 1) / p.splits) * (NTOK / 4) * 32 * 16;
    const uint32_t lq_off = static_cast<uint32_t>(quarter / p.splits) * (NTOK / 4) * 32 * 16 + lane * 16;
    const int c_lo = wa_col_lo<NTOK>(team), c_hi = c_lo + wa_ncols<NTOK>(team);
    if (warp >= 2 && prod_ok && o != split) {
      const uint32_t slot = static_cast<uint32_t>(split < o ? split : split - 1);
      for (int c = c_lo; c < c_hi && c < ncv; c += 16) {
        uint32_t v[16];
        __syncwarp();
        tmem_ld_32x32b_x16(dcol + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          st_cluster_v4(base + slot * slot_bytes + lq_off + ((c + j) >> 2) * 512u, static_cast<uint32_t>(o),
                        make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                                    __uint_as_float(v[j + 3])));
      }
    }
    cluster_sync();  // the slices have landed
    if (warp >= 2 && prod_ok && o == split) {
      const int row = n0 + quarter * 32 + lane;
      for (int c = c_lo; c < c_hi && c < ncv; c += 16) {
        uint32_t v[16];
        __syncwarp();
        tmem_ld_32x32b_x16(dcol + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int sp = 0; sp < p.splits; ++sp) {
            float4 x;
            if (sp == split) {
              x = make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]), __uint_as_float(v[j + 2]),
                              __uint_as_float(v[j + 3]));
            } else {
              const uint32_t slot = static_cast<uint32_t>(sp < split ? sp : sp - 1);
              x = *reinterpret_cast<const float4*>(smem + slot * slot_bytes + lq_off + ((c + j) >> 2) * 512u);
            }
            if (sp == 0) {
              sum = x;
            } else {
              sum.x += x.x;
              sum.y += x.y;
              sum.z += x.z;
              sum.w += x.w;
            }
          }
          if (row < p.N) {
            const float f[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = tok0 + c + j + e;
              if (tok < p.M) p.y[static_cast<int64_t>(tok) * p.N + row] = __float2bfloat16_rn(f[e]);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, Cfg::kTmemCols);
  }
}

// ====================================================================== backward dX
struct WbParams {
  const uint8_t* codes;
  const int8_t* absq;
  const float* step;
  const float* mean;
  __nv_bfloat16* dx;  // [M, K]
  unsigned* status;
  int M, N, K, r;
  int lora_blocks, accumulate;
  // the n blocks of a tile are split over `splits` CTAs, one cluster (the last also runs the LoRA
  // steps); their float32 results are added through distributed shared memory
  int splits, nb_per_split;
  unsigned long long wait_ns;
};

constexpr int kWbTeamThreads = 256;  // one team decodes a whole [64 n x 256 k] block: one 64-weight unit per thread
constexpr int kWbThreads = 64 + 2 * kWbTeamThreads;  // warp 0 TMA + TMEM, warp 1 MMA, two producer teams
constexpr uint32_t kWbABytes = 256 * 128;      // 256 tokens x 64 n, bf16 (two M = 128 halves)
constexpr uint32_t kWbBBytes = 4 * 64 * 128;   // 4 slabs of [64 n rows x 64 k]
constexpr uint32_t kWbStage = kWbABytes + kWbBBytes;

template <int STAGES>
struct WbCfg {
  static constexpr size_t kSmem = 1024 + STAGES * kWbStage + (2 * STAGES + 1) * 8 + 16;
};

// Tile: 256 tokens x 256 output columns.  Each dequantised W block [64 n x 256 k]
// feeds two M = 128 MMAs (tokens 0..127 and 128..255) into two TMEM
// accumulators (columns 0..255 and 256..511), so the decode is shared by 256 tokens.
template <int STAGES>
__global__ void __launch_bounds__(kWbThreads, 1)
    k_qgemm_wb(const __grid_constant__ CUtensorMap tm_dy, const __grid_constant__ CUtensorMap tm_su,
               const __grid_constant__ CUtensorMap tm_la, const WbParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * kWbStage);
  uint64_t* empty = full + STAGES;
  uint64_t* acc_full = empty + STAGES;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  volatile int* vabort = abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // split = this CTA's rank in its cluster (clusters of `splits` CTAs along z)
  const int k0 = blockIdx.x * 256, tok0 = blockIdx.y * 256, split = blockIdx.z;
  // this CTA's n blocks [nb0, nb0 + n_main); the last split also runs the LoRA k steps
  const int nb0 = split * p.nb_per_split;
  const int n_main = min((p.N + 63) / 64 - nb0, p.nb_per_split);
  const int n_iter = n_main + (split == p.splits - 1 ? p.lora_blocks : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1 + kWbTeamThreads);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_holder, 512);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;
  bool prod_ok = false;  // producers: the accumulators hold this CTA's result

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_dy);
      tma_prefetch_desc(&tm_su);
      tma_prefetch_desc(&tm_la);
      for (int i = 0; i < n_iter; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); break; }
        uint8_t* sa = smem + s * kWbStage;
        if (i < n_main) {
          mbar_arrive_expect_tx(&full[s], kWbABytes);
          tma_load_2d(sa, &tm_dy, &full[s], (nb0 + i) * 64, tok0);
        } else {
          const int e = i - n_main;
          if (e == 0) griddep_wait();  // sU is written by the preceding LoRA down kernel
          mbar_arrive_expect_tx(&full[s], kWbStage);
          tma_load_2d(sa, &tm_su, &full[s], e * 64, tok0);
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) tma_load_2d(sa + kWbABytes + sl * 8192, &tm_la, &full[s], k0 + sl * 64, e * 64);
        }
      }
      // no LoRA k steps: still wait once for the preceding kernel, so this grid never completes
      // before it does (later kernels of the stream rely on that order)
      if (n_iter == n_main) griddep_wait();
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 256, 0, 1);
      for (int i = 0; i < n_iter; ++i) {
        const int s = i % STAGES;
        const uint32_t ph = (i / STAGES) & 1;
        if (!mbar_wait(&full[s], ph, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); break; }
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + s * kWbStage);
        const uint32_t b_addr = a_addr + kWbABytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bdesc = sdesc_sw128(b_addr + kk * 2048, 8192, 1024);
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          mma_bf16_ss(tbase, sdesc_sw128(a_addr + kk * 32, 16, 1024), bdesc, idesc, acc);
          mma_bf16_ss(tbase + 256, sdesc_sw128(a_addr + 128 * 128 + kk * 32, 16, 1024), bdesc, idesc, acc);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(acc_full);
    }
  } else {
    // ---------------------------------------------------------------- producers
    const int team = (warp - 2) >> 3;                    // 0 or 1: k blocks of this parity
    const int t = ((warp - 2) & 7) * 32 + lane;          // 0..255: unit within the block
    const uint32_t rrow = t & 63, slab = t >> 6;         // weight row n - 64 i, 64-wide k slab
    const float mu = *p.mean;
    const int kb_row = p.K / 64;
    const int kblk = (k0 >> 6) + slab;
    // the codes and absmax of a unit are loaded one trip ahead of its decode
    uint4 nc0 = make_uint4(0, 0, 0, 0), nc1 = nc0;
    int8_t nq = 0;
    float nstep = 0.f;
    auto fetch = [&](int i) {
      const int n = (nb0 + i) * 64 + rrow;
      if (i < n_main && n < p.N && kblk < kb_row) {
        const uint8_t* cp = p.codes + static_cast<int64_t>(n) * (p.K / 2) + kblk * 32;
        nc0 = ldg_nc_v4(cp);
        nc1 = ldg_nc_v4(cp + 16);
        const int64_t ai = static_cast<int64_t>(n) * kb_row + kblk;
        nq = p.absq[ai];
        nstep = p.step[ai >> 8];
      }
    };
    fetch(team);
    bool alive = true;
    for (int i = team; i < n_iter && alive; i += 2) {
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      const bool is_main = i < n_main;
      const int n = (nb0 + i) * 64 + rrow;
      const bool uok = is_main && (n < p.N) && (kblk < kb_row);
      const uint4 c0 = nc0, c1 = nc1;
      const float a2 = restore_absmax(nq, nstep, mu);
      fetch(i + 2);
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ph ^ 1, p.wait_ns, vabort));
      if (!ok) { if (lane == 0) abort_cta(p.status, abort_flag); alive = false; break; }
      if (is_main) {
        uint32_t words[32];
        if (uok) {
          nf4_decode_block(c0, c1, a2, words);
        } else {
#pragma unroll
          for (int q = 0; q < 32; ++q) words[q] = 0;
        }
        const uint32_t slab_base = smem_u32(smem + s * kWbStage + kWbABytes) + slab * 8192;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          sts_v4(slab_base + sw128_offset(rrow, ch), words[4 * ch], words[4 * ch + 1], words[4 * ch + 2],
                 words[4 * ch + 3]);
        fence_proxy_async_smem();
      }
      mbar_arrive(&full[s]);
    }
    // ---------------------------------------------------------------- epilogue
    // the four warps of each TMEM lane quarter share its 2 accumulators x 8 column chunks
    bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, p.wait_ns, vabort));
    ok = ok && !*vabort;
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    prod_ok = ok;
    const int quarter = warp & 3;
    const int wq = (warp - 2) >> 2;  // 0..3 among the warps of this quarter
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    if (ok && p.splits == 1) {
      for (int chunk = wq; chunk < 16; chunk += 4) {
        const int acc = chunk >> 3, col = (chunk & 7) * 32;
        const int tok = tok0 + acc * 128 + quarter * 32 + lane;
        uint32_t v[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tbase + lane_field + acc * 256 + col, v);
        tmem_ld_wait();
        const int kc = k0 + col;
        if (tok < p.M && kc < p.K) {
          uint4* dst = reinterpret_cast<uint4*>(p.dx + static_cast<int64_t>(tok) * p.K + kc);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(v[8 * q + j]);
            if (p.accumulate) {
              const uint4 old = dst[q];
              const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                f[2 * j] += __uint_as_float(ow[j] << 16);
                f[2 * j + 1] += __uint_as_float(ow[j] & 0xffff0000u);
              }
            }
            dst[q] = make_uint4(pack_bf16x2_rn(f[0], f[1]), pack_bf16x2_rn(f[2], f[3]), pack_bf16x2_rn(f[4], f[5]),
                                pack_bf16x2_rn(f[6], f[7]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (p.splits > 1) {
    // Split n: the tile's 8 chunks of 32 output columns are owned round-robin (chunk c by the CTA
    // of cluster rank c % splits).  Each CTA sends every chunk it does not own, as float32 values of
    // both accumulators, to the owner's now idle stage buffers -- slot s (s - 1 past the owner) for
    // sender s, laid out [owned chunk c / splits][accumulator][8 groups of 4 columns][128 rows]
    // float4, over the accumulators that hold tokens -- and each owner adds the splits' values in
    // split order and writes dX.
    tc_fence_after();
    cluster_sync();  // every CTA of the cluster is past its k loop: the stage buffers are free
    const int ntok = min(256, p.M - tok0);
    const int quarter = warp & 3, wq = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t base = smem_u32(smem);
    const int nacc = ntok > 128 ? 2 : 1;  // accumulators holding tokens
    const uint32_t slot_bytes = static_cast<uint32_t>((8 + p.splits - 1) / p.splits * nacc) * (8 * 128 * 16);
    // unit u = (accumulator u >> 3, chunk u & 7); a warp takes the units u = wq (mod 4)
    auto unit_kept = [&](int acc, int cc) { return acc * 128 < ntok && k0 + 32 * cc < p.K; };
    if (warp >= 2 && prod_ok) {
      for (int u = wq; u < 16; u += 4) {
        const int acc = u >> 3, cc = u & 7, o = cc % p.splits;
        if (o == split || !unit_kept(acc, cc)) continue;  // warp-uniform
        uint32_t v[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tbase + lane_field + acc * 256 + 32 * cc, v);
        tmem_ld_wait();
        const uint32_t slot = static_cast<uint32_t>(split < o ? split : split - 1);
        const uint32_t at = base + slot * slot_bytes + static_cast<uint32_t>(((cc / p.splits) * nacc + acc) * 8) * 2048u +
                            static_cast<uint32_t>(row) * 16u;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          st_cluster_v4(at + q * 2048u, static_cast<uint32_t>(o),
                        make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                    __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3])));
      }
    }
    cluster_sync();  // the slots have landed
    if (warp >= 2 && prod_ok) {
      for (int u = wq; u < 16; u += 4) {
        const int acc = u >> 3, cc = u & 7;
        if (cc % p.splits != split || !unit_kept(acc, cc)) continue;  // warp-uniform
        uint32_t v[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tbase + lane_field + acc * 256 + 32 * cc, v);
        tmem_ld_wait();
        const int tl = acc * 128 + row;
        if (tl >= ntok) continue;
        const uint32_t in_slot = static_cast<uint32_t>(((cc / p.splits) * nacc + acc) * 8) * 2048u +
                                 static_cast<uint32_t>(row) * 16u;
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {  // 8 columns per 16-byte store
          float f[8];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int q = 2 * q8 + h;
            float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sp = 0; sp < p.splits; ++sp) {
              float4 x;
              if (sp == split) {
                x = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                                __uint_as_float(v[4 * q + 3]));
              } else {
                const uint32_t slot = static_cast<uint32_t>(sp < split ? sp : sp - 1);
                x = *reinterpret_cast<const float4*>(smem + slot * slot_bytes + in_slot + q * 2048u);
              }
              if (sp == 0) {
                sum = x;
              } else {
                sum.x += x.x;
                sum.y += x.y;
                sum.z += x.z;
                sum.w += x.w;
              }
            }
            f[4 * h] = sum.x;
            f[4 * h + 1] = sum.y;
            f[4 * h + 2] = sum.z;
            f[4 * h + 3] = sum.w;
          }
          uint4* dst = reinterpret_cast<uint4*>(p.dx + static_cast<int64_t>(tok0 + tl) * p.K + k0 + 32 * cc + 8 * q8);
          if (p.accumulate) {
            const uint4 old = *dst;
            const uint32_t ow[4] = {old.x, old.y, old.z, old.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              f[2 * j] += __uint_as_float(ow[j] << 16);
              f[2 * j + 1] += __uint_as_float(ow[j] & 0xffff0000u);
            }
          }
          *dst = make_uint4(pack_bf16x2_rn(f[0], f[1]), pack_bf16x2_rn(f[2], f[3]), pack_bf16x2_rn(f[4], f[5]),
                            pack_bf16x2_rn(f[6], f[7]));
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ====================================================================== LoRA gradients
struct LgParams {
  float* da;  // [r, K]
  float* db;  // [N, r]
  unsigned* status;
  int M, N, K, r;
  int tiles_a, tiles;  // 128-column tiles of dA^T (first tiles_a) and of dB
  int accum_da, accum_db;
  float da_scale;      // dA = da_scale * (sU^T X); 1 except under dropout
  unsigned long long wait_ns;
};

constexpr int kLgThreads = 192;  // warp 0 TMA + TMEM, warp 1 MMA, warps 2..5 epilogue

template <int RP>  // MMA N: 64 or 128
struct LgCfg {
  static constexpr uint32_t kABytes = 2 * 8192;           // [64 m x 128 c] as two 64-wide slabs
  static constexpr uint32_t kBBytes = (RP / 64) * 8192;   // [64 m x RP j]
  static constexpr uint32_t kStage = kABytes + kBBytes;
  static constexpr int kStages = RP == 64 ? 8 : 6;        // deep ring: few CTAs stream every token
  static constexpr uint32_t kTmemCols = 2 * RP;           // double-buffered accumulator
  static constexpr size_t kSmem = 1024 + kStages * kStage + (2 * kStages + 4) * 8 + 16;
};

// Persistent: CTA b takes column tiles b, b + gridDim.x, ...; for each, all
// tokens stream through the TMA ring (no cross-CTA reduction: deterministic).
template <int RP>
__global__ void __launch_bounds__(kLgThreads, 1)
    k_lora_grad(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                const __grid_constant__ CUtensorMap tm_su, const __grid_constant__ CUtensorMap tm_st,
                const LgParams p) {
  using Cfg = LgCfg<RP>;
  constexpr int kLgStages = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kLgStages * Cfg::kStage);
  uint64_t* empty = full + kLgStages;
  uint64_t* acc_full = empty + kLgStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;      // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  volatile int* vabort = abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_iter = (p.M + 63) / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kLgStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_holder, Cfg::kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      griddep_wait();  // sU and sT come from the preceding kernel
      // the kernels that follow may start launching now (every kernel before this one has completed)
      griddep_launch_dependents();
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_dy);
      int g = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x) {
        const bool is_b = tile >= p.tiles_a;
        const int c0 = (is_b ? tile - p.tiles_a : tile) * 128;
        const CUtensorMap* tq = is_b ? &tm_dy : &tm_x;
        const CUtensorMap* tp = is_b ? &tm_st : &tm_su;
        for (int i = 0; i < n_iter; ++i, ++g) {
          const int s = g % kLgStages;
          const uint32_t ph = (g / kLgStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); ok = false; break; }
          uint8_t* sa = smem + s * Cfg::kStage;
          mbar_arrive_expect_tx(&full[s], Cfg::kStage);
          tma_load_2d(sa, tq, &full[s], c0, i * 64);
          tma_load_2d(sa + 8192, tq, &full[s], c0 + 64, i * 64);
#pragma unroll
          for (int sl = 0; sl < RP / 64; ++sl) tma_load_2d(sa + Cfg::kABytes + sl * 8192, tp, &full[s], sl * 64, i * 64);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, RP, 1, 1);
      int g = 0, j = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.tiles && ok; tile += gridDim.x, ++j) {
        const int buf = j & 1;
        if (!mbar_wait(&acc_empty[buf], ((j >> 1) & 1) ^ 1, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); break; }
        tc_fence_after();
        for (int i = 0; i < n_iter; ++i, ++g) {
          const int s = g % kLgStages;
          const uint32_t ph = (g / kLgStages) & 1;
          if (!mbar_wait(&full[s], ph, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + s * Cfg::kStage);
          const uint32_t b_addr = a_addr + Cfg::kABytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = sdesc_sw128(a_addr + kk * 2048, 8192, 1024);
            const uint64_t bdesc = sdesc_sw128(b_addr + kk * 2048, 8192, 1024);
            mma_bf16_ss(tbase + buf * RP, adesc, bdesc, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&acc_full[buf]);
      }
    }
  } else {
    const int quarter = warp & 3;
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    int j = 0;
    for (int tile = blockIdx.x; tile < p.tiles; tile += gridDim.x, ++j) {
      const int buf = j & 1;
      bool ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (j >> 1) & 1, p.wait_ns, vabort));
      ok = __all_sync(0xffffffffu, ok && !*vabort);
      if (!ok) break;
      tc_fence_after();
      const bool is_b = tile >= p.tiles_a;
      const int c = (is_b ? tile - p.tiles_a : tile) * 128 + quarter * 32 + lane;
      const int C = is_b ? p.N : p.K;
      for (int j0 = 0; j0 < RP && j0 < p.r; j0 += 16) {
        uint32_t v[16];
        __syncwarp();
        tmem_ld_32x32b_x16(tbase + lane_field + buf * RP + j0, v);
        tmem_ld_wait();
        if (c < C) {
          if (!is_b) {
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
              if (j0 + jj >= p.r) break;
              float* d = p.da + static_cast<int64_t>(j0 + jj) * p.K + c;
              const float val = __fmul_rn(__uint_as_float(v[jj]), p.da_scale);
              *d = p.accum_da ? (*d + val) : val;
            }
          } else {
            float* d = p.db + static_cast<int64_t>(c) * p.r + j0;
            if ((p.r & 3) == 0) {  // rows of dB start on 16-byte boundaries: 4 floats at a time
#pragma unroll
              for (int jj = 0; jj < 16; jj += 4) {
                if (j0 + jj >= p.r) break;
                float4 val = make_float4(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1]),
                                         __uint_as_float(v[jj + 2]), __uint_as_float(v[jj + 3]));
                if (p.accum_db) {
                  const float4 o = *reinterpret_cast<const float4*>(d + jj);
                  val.x += o.x; val.y += o.y; val.z += o.z; val.w += o.w;
                }
                *reinterpret_cast<float4*>(d + jj) = val;
              }
            } else {
#pragma unroll
              for (int jj = 0; jj < 16; ++jj) {
                if (j0 + jj >= p.r) break;
                const float val = __uint_as_float(v[jj]);
                d[jj] = p.accum_db ? d[jj] + val : val;
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tbase, Cfg::kTmemCols);
  }
}

// ====================================================================== bounded-wait self test
__global__ void k_wait_selftest(unsigned* status, unsigned long long wait_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, wait_ns, nullptr)) latch_status(status, ST_TIMEOUT);
}

// ====================================================================== host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;
static char g_tm_err[256] = "";

const char* tensor_map_error() { return g_tm_err; }

static bool get_encode() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    const cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      snprintf(g_tm_err, sizeof(g_tm_err), "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(e));
  });
  return g_encode != nullptr;
}

// bf16 matrix [outer, inner] with row pitch `pitch` bytes; box [box_outer, box_inner]; 128-byte swizzle.
bool make_tensor_map_bf16_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t pitch,
                    uint32_t box_inner, uint32_t box_outer) {
  if (!get_encode()) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_tm_err, sizeof(g_tm_err), "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu] pitch %llu", (int)r,
             (unsigned long long)outer, (unsigned long long)inner, (unsigned long long)pitch);
    return false;
  }
  return true;
}

struct FwdPlan {
  int ntok, row_tiles, tok_tiles, splits, kb_per_split;
};

static FwdPlan plan_fwd(int M, int N, int K, int num_sms) {
  FwdPlan pl;
  if (M < 1) M = 1;
  if (num_sms < 1) num_sms = 1;
  pl.ntok = M <= 16 ? 16 : (M <= 64 ? 64 : (M <= 128 ? 128 : 256));
  pl.row_tiles = (N + 127) / 128;
  pl.tok_tiles = (M + pl.ntok - 1) / pl.ntok;
  const int tiles = pl.row_tiles * pl.tok_tiles;
  const int kb_total = K / 64;
  // split k while the grid still fits one wave (one 576-thread CTA per SM); the splits of a tile
  // form one cluster and add their partials through distributed shared memory
  int splits = num_sms / tiles;
  if (splits > kMaxSplitK) splits = kMaxSplitK;
  if (splits > kb_total) splits = kb_total;
  if (splits < 1) splits = 1;
  pl.kb_per_split = (kb_total + splits - 1) / splits;
  pl.splits = (kb_total + pl.kb_per_split - 1) / pl.kb_per_split;
  return pl;
}

struct BwdPlan {
  int ktiles, tok_tiles, splits, nb_per_split;
};

// Backward dX: 256-column x 256-token tiles; with few tiles (small token counts) the n blocks of
// a tile are split over up to 4 CTAs of a cluster while the grid fits one wave.
static BwdPlan plan_bwd(int M, int N, int K, int num_sms) {
  BwdPlan pl;
  if (M < 1) M = 1;
  if (num_sms < 1) num_sms = 1;
  pl.ktiles = (K + 255) / 256;
  pl.tok_tiles = (M + 255) / 256;
  const int tiles = pl.ktiles * pl.tok_tiles, nb = (N + 63) / 64 > 0 ? (N + 63) / 64 : 1;
  int splits = num_sms / tiles;
  if (splits > kMaxSplitK) splits = kMaxSplitK;
  if (splits > nb) splits = nb;
  if (splits < 1) splits = 1;
  pl.nb_per_split = (nb + splits - 1) / splits;
  pl.splits = (nb + pl.nb_per_split - 1) / pl.nb_per_split;
  return pl;
}

size_t bwd_gemm_workspace_bytes(int M, int N, int K, int num_sms) {
  (void)M, (void)N, (void)K, (void)num_sms;
  return 0;  // split n adds its partials inside a cluster
}

size_t fwd_gemm_workspace_bytes(int M, int N, int K, int num_sms) {
  (void)M, (void)N, (void)K, (void)num_sms;
  return 0;  // split k adds its partials inside a cluster
}

// Launch with programmatic stream serialization: the kernel may start while the
// preceding kernel of the stream (the LoRA down-projection) still runs; it
// waits for it (griddep_wait) only before loading that kernel's output.
// `cluster` > 1: clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl_z(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                int cluster, int cluster_z, Args&&... args);
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              int cluster, Args&&... args) {
  return launch_pdl_z(kernel, grid, block, smem, s, cluster, 1, std::forward<Args>(args)...);
}
// `cluster` > 1: clusters of that many CTAs along x; `cluster_z` > 1: along z.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl_z(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                int cluster, int cluster_z, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = cluster_z;
  cfg.attrs = attr;
  cfg.numAttrs = (cluster > 1 || cluster_z > 1) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int NTOK, int STAGES>
static cudaError_t run_wa(const CUtensorMap& tx, const CUtensorMap& tst, const WaParams& prm, dim3 grid,
                          cudaStream_t s) {
  using Cfg = WaCfg<NTOK, STAGES>;
  cudaError_t e = set_smem_limit_once(k_qgemm_wa<NTOK, STAGES>, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  e = launch_pdl_z(k_qgemm_wa<NTOK, STAGES>, grid, dim3(kWaThreads), Cfg::kSmem, s, 1, static_cast<int>(grid.z), tx,
                   tst, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_fwd_gemm(const __nv_bfloat16* x, int M, const Nf4Dev& w, const __nv_bfloat16* st,
                            const __nv_bfloat16* lora_b, int r, __nv_bfloat16* y, void* ws, unsigned* status,
                            uint64_t wait_ns, int num_sms, cudaStream_t s) {
  if (use_pair_gemm(M)) return launch_fwd_gemm_pair(x, M, w, st, lora_b, r, y, status, wait_ns, s);
  const int N = static_cast<int>(w.n), K = static_cast<int>(w.k);
  const FwdPlan pl = plan_fwd(M, N, K, num_sms);
  CUtensorMap tx, tst;
  if (!make_tensor_map_bf16_2d(&tx, x, K, M, static_cast<uint64_t>(K) * 2, 64, pl.ntok)) return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tst, st, lora_ld(r), M, static_cast<uint64_t>(lora_ld(r)) * 2, 64, pl.ntok))
    return cudaErrorInvalidValue;
  WaParams prm;
  prm.codes = w.codes;
  prm.absq = w.absq;
  prm.step = w.step;
  prm.mean = w.mean;
  prm.lora_b = lora_b;
  prm.y = y;
  prm.status = status;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.r = r;
  prm.kb_per_split = pl.kb_per_split;
  prm.splits = pl.splits;
  prm.lora_blocks = (r + 63) / 64;
  prm.wait_ns = wait_ns;
  (void)ws;
  const dim3 grid(pl.row_tiles, pl.tok_tiles, pl.splits);  // the splits of a tile form one cluster
  if (pl.ntok == 16) return run_wa<16, 4>(tx, tst, prm, grid, s);
  if (pl.ntok == 64) return run_wa<64, 4>(tx, tst, prm, grid, s);
  if (pl.ntok == 128) return run_wa<128, 4>(tx, tst, prm, grid, s);
  return run_wa<256, 4>(tx, tst, prm, grid, s);
}

cudaError_t launch_bwd_dx_gemm(const __nv_bfloat16* dy, int M, const Nf4Dev& w, const __nv_bfloat16* su,
                               const __nv_bfloat16* lora_a, int r, __nv_bfloat16* dx, int accumulate, void* ws,
                               unsigned* status, uint64_t wait_ns, int num_sms, cudaStream_t s, int with_lora) {
  if (use_pair_gemm(M))
    return launch_bwd_gemm_pair(dy, M, w, su, lora_a, r, dx, accumulate, status, wait_ns, s, with_lora);
  const int N = static_cast<int>(w.n), K = static_cast<int>(w.k);
  CUtensorMap tdy, tsu, tla;
  if (!make_tensor_map_bf16_2d(&tdy, dy, N, M, static_cast<uint64_t>(N) * 2, 64, 256)) return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tsu, su, lora_ld(r), M, static_cast<uint64_t>(lora_ld(r)) * 2, 64, 256))
    return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tla, lora_a, K, r, static_cast<uint64_t>(K) * 2, 64, 64)) return cudaErrorInvalidValue;
  WbParams prm;
  prm.codes = w.codes;
  prm.absq = w.absq;
  prm.step = w.step;
  prm.mean = w.mean;
  prm.dx = dx;
  prm.status = status;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.r = r;
  prm.lora_blocks = with_lora ? (r + 63) / 64 : 0;
  prm.accumulate = accumulate;
  prm.wait_ns = wait_ns;
  const BwdPlan pl = plan_bwd(M, N, K, num_sms);
  prm.splits = pl.splits;
  prm.nb_per_split = pl.nb_per_split;
  (void)ws;
  constexpr int kStages = 3;
  const size_t smem = WbCfg<kStages>::kSmem;
  cudaError_t e = set_smem_limit_once(k_qgemm_wb<kStages>, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(pl.ktiles, pl.tok_tiles, pl.splits);
  e = launch_pdl_z(k_qgemm_wb<kStages>, grid, dim3(kWbThreads), smem, s, 1, pl.splits, tdy, tsu, tla, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

size_t lora_grads_workspace_bytes(int M, int N, int K, int r, int num_sms) {
  (void)M, (void)N, (void)K, (void)r, (void)num_sms;
  return 0;  // no cross-CTA reduction
}

cudaError_t launch_lora_grads(const __nv_bfloat16* x, const __nv_bfloat16* dy, const __nv_bfloat16* su,
                              const __nv_bfloat16* st, int M, int N, int K, int r, float* da, float* db,
                              int accum_da, int accum_db, void* ws, unsigned* status, uint64_t wait_ns, int max_ctas,
                              cudaStream_t s, float da_scale) {
  (void)ws;
  CUtensorMap tx, tdy, tsu, tst;
  if (!make_tensor_map_bf16_2d(&tx, x, K, M, static_cast<uint64_t>(K) * 2, 64, 64)) return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tdy, dy, N, M, static_cast<uint64_t>(N) * 2, 64, 64)) return cudaErrorInvalidValue;
  const uint64_t rk = static_cast<uint64_t>(lora_ld(r));
  if (!make_tensor_map_bf16_2d(&tsu, su, rk, M, rk * 2, 64, 64)) return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tst, st, rk, M, rk * 2, 64, 64)) return cudaErrorInvalidValue;
  LgParams prm;
  prm.da = da;
  prm.db = db;
  prm.status = status;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.r = r;
  prm.tiles_a = (K + 127) / 128;
  prm.tiles = prm.tiles_a + (N + 127) / 128;
  prm.accum_da = accum_da;
  prm.accum_db = accum_db;
  prm.da_scale = da_scale;
  prm.wait_ns = wait_ns;
  int grid = prm.tiles < max_ctas ? prm.tiles : max_ctas;
  if (grid >= 2) grid &= ~1;  // clusters of two: the CTAs sit on whole TPCs, which the pair GEMMs need
  if (grid < 1) grid = 1;
  const int cluster = grid >= 2 ? 2 : 1;
  cudaError_t e;
  if (r <= 64) {
    e = set_smem_limit_once(k_lora_grad<64>, LgCfg<64>::kSmem);
    if (e == cudaSuccess) e = launch_pdl(k_lora_grad<64>, dim3(grid), dim3(kLgThreads), LgCfg<64>::kSmem, s, cluster, tx, tdy, tsu, tst, prm);
  } else {
    e = set_smem_limit_once(k_lora_grad<128>, LgCfg<128>::kSmem);
    if (e == cudaSuccess) e = launch_pdl(k_lora_grad<128>, dim3(grid), dim3(kLgThreads), LgCfg<128>::kSmem, s, cluster, tx, tdy, tsu, tst, prm);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// SMs a GEMM grid leaves idle in its last wave: the budget for the side kernels
// that run beside it (all of them when the grid fills its waves exactly).
int idle_sms_beside(int gemm_ctas, int num_sms) {
  const int rem = gemm_ctas % num_sms;
  const int idle = rem == 0 ? 0 : num_sms - rem;
  return idle >= 8 ? idle : num_sms;
}

int fwd_gemm_ctas(int M, int N, int K, int num_sms) {
  if (use_pair_gemm(M)) return fwd_pair_ctas(M, N);
  const FwdPlan pl = plan_fwd(M, N, K, num_sms);
  return pl.row_tiles * pl.tok_tiles * pl.splits;
}

int bwd_gemm_ctas(int M, int N, int K, int num_sms) {
  if (use_pair_gemm(M)) return bwd_pair_ctas(M, K);
  const BwdPlan pl = plan_bwd(M, N, K, num_sms);
  return pl.ktiles * pl.tok_tiles * pl.splits;
}

cudaError_t launch_wait_selftest(unsigned* status, uint64_t wait_ns, cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>(status, wait_ns);
  return cudaGetLastError();
}

}  // namespace qlora
