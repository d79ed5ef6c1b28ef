// NF4 QLoRA GEMMs on CTA pairs (tcgen05 cta_group::2), for token counts > 256.
//
// The frozen product of the QLoRA linear (glossary "QLoRA", "How QLoRA works":
// the NF4 weight is dequantised to bfloat16 for the matmul, the LoRA output is
// added; Day 25 notes "Fine-tuning and LoRA/QLoRA", section 2.1, scaled by
// s = alpha / r as in section 6.2):
//
//   forward   D[n, m] = sum_k deq(W)[n, k] X[m, k]  + sum_j B[n, j] sT[m, j]      (Y = D^T)
//   backward  D[m, k] = sum_n dY[m, n] deq(W)[n, k] + sum_j sU[m, j] A[j, k]      (dX = D)
//
// The dequantisation runs on the ALU pipe (about four integer ops per weight),
// so a decoded weight has to feed enough MMA work to keep it off the critical
// path: each pair of CTAs decodes a [256 x 64] slice of W per k step and uses it
// for 512 tokens (two M = 256 x N = 256 accumulators, 512 TMEM columns per CTA).
// The MMA reads both operands from shared memory; with the pair each SM reads
// its own A half and its own B half, about 64 B/clk at the tensor rate, plus
// 48 KB of stage fills per 1024 MMA cycles.
//
// Roles per CTA (576 threads): warp 0 lane 0 = TMA (activations), warp 0 =
// TMEM allocation; warp 1 lane 0 of the even CTA = MMA issue; warps 2..17 =
// four producer teams (k steps round-robin) that decode one W slice each into
// shared memory (or copy the LoRA rows for the last k steps), then the epilogue.
//
// Stage (48 KB): [0, 32K) two TMA boxes [128 rows x 64] bf16 (one per
// accumulator), K-major 128B swizzle; [32K, 48K) the CTA's decoded W tile:
//   forward  A operand, K-major: 128 W rows x 64 k;
//   backward B operand, MN-major: 64 n rows x 128 output columns (two 64-wide slabs).
// "Stage s full" is one barrier in the even CTA that both CTAs complete: the odd
// CTA's TMA signals it across the pair and its producer warps arrive remotely,
// so the MMA thread waits once per k step.  "Stage s empty" lives in both CTAs
// and is released by one multicast MMA commit.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

struct PairParams {
  const uint8_t* codes;
  const int8_t* absq;
  const float* step;
  const float* mean;
  const __nv_bfloat16* lora_b;  // forward: [N, r]
  const __nv_bfloat16* lora_a;  // backward: [r, K]
  __nv_bfloat16* out;           // forward: Y [M, N]; backward: dX [M, K]
  unsigned* status;
  int M, N, K, r;
  int lora_blocks, accumulate;
  int staged_store;  // write the result through shared memory with TMA stores (tm_out)
  unsigned long long wait_ns;
};

constexpr int kPrTeams = 4;
constexpr int kPrThreads = 64 + kPrTeams * 128;
constexpr int kPrStages = kPrTeams;                 // team t always fills stage t
constexpr uint32_t kPrBox = 128 * 128;              // [128 rows x 64] bf16
constexpr uint32_t kPrActBytes = 2 * kPrBox;        // one box per accumulator
constexpr uint32_t kPrProdBytes = 16384;            // decoded W tile of this CTA
constexpr uint32_t kPrStage = kPrActBytes + kPrProdBytes;
constexpr uint32_t kPrBarBase = kPrStages * kPrStage;
constexpr int kPrBars = 2 * kPrStages + 1;
constexpr size_t kPrSmem = 1024 + kPrBarBase + kPrBars * 8 + 16;
static_assert(kPrSmem <= 232448, "dynamic shared memory per block");
constexpr int kPrTokens = 512;  // tokens per pair tile
constexpr int kPrCols = 256;    // W rows (forward) / output columns (backward) per pair tile

// TMA load whose completion is signalled on a barrier of the even CTA of the
// pair (`bar_cluster` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_to_pair_bar(void* smem_dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                        int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
      : "memory");
}
// Tiled TMA store of one box from shared memory; the copy is clipped to the tensor.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t smem_src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(smem_src)
               : "memory");
}
// Wait until the issued TMA stores have read their shared-memory sources.
__device__ __forceinline__ void tma_store_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  return ra;
}
__device__ __forceinline__ void mbar_arrive_cluster_addr(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

template <bool BWD>
__global__ void __launch_bounds__(kPrThreads, 1)
    k_qgemm_pair(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_low,
                 const __grid_constant__ CUtensorMap tm_out, const PairParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPrBarBase);  // used in the even CTA
  uint64_t* empty = full + kPrStages;
  uint64_t* acc_full = empty + kPrStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_full + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  volatile int* vabort = abort_flag;

  const uint32_t rank = cluster_ctarank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x >> 1;
  const int tok0 = blockIdx.y * kPrTokens;
  const int n_main = BWD ? (p.N + 63) / 64 : p.K / 64;
  const int n_iter = n_main + p.lora_blocks;

  // producer unit of this thread (warps 2..17); its first codes are fetched before the set-up
  const int team = (warp - 2) >> 2;
  const int t = ((warp - 2) & 3) * 32 + lane;  // 0..127
  const float mu = *p.mean;
  const int kb_row = p.K / 64;
  // forward: W row n_fix (all k steps); backward: row i * 64 + rrow, k block kblk
  const int n_fix = pair * kPrCols + static_cast<int>(rank) * 128 + t;
  const uint32_t rrow = t & 63, slab = t >> 6;
  const int col0 = pair * kPrCols + static_cast<int>(rank) * 128 + static_cast<int>(slab) * 64;
  const int kblk = col0 / 64;
  uint4 nc0 = make_uint4(0, 0, 0, 0), nc1 = nc0;
  int8_t nq = 0;
  float nstep = 0.f;
  auto unit_ok = [&](int i) {
    if (i >= n_main) return false;
    return BWD ? (i * 64 + static_cast<int>(rrow) < p.N && kblk < kb_row) : (n_fix < p.N);
  };
  auto fetch = [&](int i) {  // codes and absmax of k step i, one trip ahead of the decode
    if (unit_ok(i)) {
      const int n = BWD ? i * 64 + static_cast<int>(rrow) : n_fix;
      const int kb = BWD ? kblk : i;
      const uint8_t* cp = p.codes + static_cast<int64_t>(n) * (p.K / 2) + kb * 32;
      nc0 = ldg_nc_v4(cp);
      nc1 = ldg_nc_v4(cp + 16);
      const int64_t ai = static_cast<int64_t>(n) * kb_row + kb;
      nq = p.absq[ai];
      nstep = p.step[ai >> 8];
    }
  };
  if (warp >= 2) fetch(team);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPrStages; ++s) {
      mbar_init(&full[s], 1 + 2 * 4);  // even CTA's TMA thread + the producing team's 4 warps in each CTA
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc_pair(tmem_holder, 512);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      // accumulator a holds tokens tok0 + 256 a + [0, 256), of which this CTA
      // supplies (forward: B columns, backward: A rows) 128 rank + [0, 128)
      const int ta = tok0 + static_cast<int>(rank) * 128, tb = ta + 256;
      tma_prefetch_desc(&tm_act);
      tma_prefetch_desc(&tm_low);
      for (int i = 0; i < n_iter; ++i) {
        const int s = i % kPrStages;
        const uint32_t ph = (i / kPrStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); break; }
        uint8_t* st = smem + s * kPrStage;
        const CUtensorMap* tm = &tm_act;
        int kc = i * 64;
        if (i >= n_main) {
          if (i == n_main) griddep_wait();  // sT / sU come from the preceding kernels of the stream
          tm = &tm_low;
          kc = (i - n_main) * 64;
        }
        if (rank == 0) {
          mbar_arrive_expect_tx(&full[s], 2 * kPrActBytes);  // both CTAs' boxes
          tma_load_2d(st, tm, &full[s], kc, ta);
          tma_load_2d(st + kPrBox, tm, &full[s], kc, tb);
        } else {
          const uint32_t bar = cluster_addr(&full[s], 0);
          tma_load_2d_to_pair_bar(st, tm, bar, kc, ta);
          tma_load_2d_to_pair_bar(st + kPrBox, tm, bar, kc, tb);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(256, 256, 0, BWD ? 1 : 0);
      for (int i = 0; i < n_iter; ++i) {
        const int s = i % kPrStages;
        const uint32_t ph = (i / kPrStages) & 1;
        if (!mbar_wait<true>(&full[s], ph, p.wait_ns, vabort)) {
          abort_cta(p.status, abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t act = smem_u32(smem + s * kPrStage);
        const uint32_t prod = act + kPrActBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            uint64_t ad, bd;
            if (BWD) {
              ad = sdesc_sw128(act + a * kPrBox + kk * 32, 16, 1024);
              bd = sdesc_sw128(prod + kk * 2048, 8192, 1024);
            } else {
              ad = sdesc_sw128(prod + kk * 32, 16, 1024);
              bd = sdesc_sw128(act + a * kPrBox + kk * 32, 16, 1024);
            }
            mma_pair_bf16_ss(tbase + a * 256, ad, bd, idesc, (i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_pair_commit_multicast(&empty[s], 3);
      }
      mma_pair_commit_multicast(acc_full, 3);  // also drains the issued MMAs after an abort
    }
  } else {
    // ---------------------------------------------------------------- producers
    const uint32_t full_remote = cluster_addr(&full[team], 0);  // team t fills stage t
    bool alive = true;
    for (int i = team; i < n_iter && alive; i += kPrTeams) {
      const int sp = i % kPrStages;
      const uint32_t php = (i / kPrStages) & 1;
      uint32_t words[32];
      if (i < n_main) {
        const bool ok = unit_ok(i);
        const uint4 c0 = nc0, c1 = nc1;
        const float a2 = restore_absmax(nq, nstep, mu);
        fetch(i + kPrTeams);
        if (ok) {
          nf4_decode_block(c0, c1, a2, words);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) words[c] = 0;
        }
      } else if (!BWD) {
        // LoRA B rows: A operand row n_fix, 64 j
        const int jb = (i - n_main) * 64;
        const uint32_t* brow = reinterpret_cast<const uint32_t*>(p.lora_b + static_cast<int64_t>(n_fix) * p.r);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const int j = jb + 2 * c;
          words[c] = (n_fix < p.N && j < p.r) ? brow[j >> 1] : 0u;
        }
      } else {
        // LoRA A rows: B operand row j = jb + rrow, 64 output columns from col0
        const int j = (i - n_main) * 64 + static_cast<int>(rrow);
        const bool ok = j < p.r && col0 < p.K;  // K % 64 == 0: the 64 columns are all inside K or all past it
        const uint4* src = reinterpret_cast<const uint4*>(p.lora_a + static_cast<int64_t>(j) * p.K + col0);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint4 v = ok ? src[ch] : make_uint4(0, 0, 0, 0);
          words[4 * ch] = v.x;
          words[4 * ch + 1] = v.y;
          words[4 * ch + 2] = v.z;
          words[4 * ch + 3] = v.w;
        }
      }
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&empty[sp], php ^ 1, p.wait_ns, vabort));
      if (!ok) { if (lane == 0) abort_cta(p.status, abort_flag); alive = false; break; }
      const uint32_t base = smem_u32(smem + sp * kPrStage + kPrActBytes);
      if (BWD) {
        const uint32_t sb = base + slab * 8192;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          sts_v4(sb + sw128_offset(rrow, ch), words[4 * ch], words[4 * ch + 1], words[4 * ch + 2], words[4 * ch + 3]);
      } else {
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          sts_v4(base + sw128_offset(t, ch), words[4 * ch], words[4 * ch + 1], words[4 * ch + 2], words[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&full[sp]);
        else
          mbar_arrive_cluster_addr(full_remote);
      }
    }
    // ---------------------------------------------------------------- epilogue
    bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, p.wait_ns, vabort));
    ok = __all_sync(0xffffffffu, ok && !*vabort);
    tc_fence_after();
    const int quarter = warp & 3;  // TMEM lanes 32 quarter .. + 31
    const int wq = (warp - 2) >> 2;  // 0..3 among the warps of this lane quarter
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    const bool staged = p.staged_store && !(BWD && p.accumulate);
    // The stage buffers are free once the last MMA is done: the result is staged
    // there in 128B-swizzled boxes and written with TMA stores (clipped to M, N).
    //   forward : 4 boxes [256 tokens x 64 W rows], box (token half h, row slab q)
    //   backward: 8 boxes [128 tokens x 64 columns], box (accumulator a, column slab q)
    const uint32_t stg = smem_u32(smem);
    if (ok) {
      if (!BWD) {
        // lane = W row, column c of accumulator a = token tok0 + 256 a + c
        const int row = pair * kPrCols + static_cast<int>(rank) * 128 + quarter * 32 + lane;
        const uint32_t nn = (quarter & 1) * 32 + lane, rslab = quarter >> 1;
        for (int c = wq * 128; c < wq * 128 + 128; c += 16) {
          uint32_t v[16];
          __syncwarp();
          tmem_ld_32x32b_x16(tbase + lane_field + c, v);  // columns 256..511 are accumulator 1
          tmem_ld_wait();
          if (staged) {
            const uint32_t box = stg + ((c >> 8) * 2 + rslab) * 32768;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const uint32_t tr = (c & 255) + j;
              const uint32_t addr = box + tr * 128 + ((((nn >> 3) ^ (tr & 7)) << 4) | ((nn & 7) << 1));
              const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(v[j]));
              asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(*reinterpret_cast<const unsigned short*>(&h))
                           : "memory");
            }
          } else if (row < p.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int tok = tok0 + c + j;
              if (tok < p.M) p.out[static_cast<int64_t>(tok) * p.N + row] = __float2bfloat16_rn(__uint_as_float(v[j]));
            }
          }
        }
      } else {
        // lane = token, column c = output column pair * 256 + c
        const uint32_t tr = quarter * 32 + lane;
        for (int a = 0; a < 2; ++a) {
          const int tok = tok0 + a * 256 + static_cast<int>(rank) * 128 + static_cast<int>(tr);
          for (int c = wq * 64; c < wq * 64 + 64; c += 16) {
            uint32_t v[16];
            __syncwarp();
            tmem_ld_32x32b_x16(tbase + lane_field + a * 256 + c, v);
            tmem_ld_wait();
            float f[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(v[j]);
            const int col = pair * kPrCols + c;  // K % 64 == 0: the 16 columns are all inside K or all past it
            __nv_bfloat16* d = p.out + static_cast<int64_t>(tok) * p.K + col;
            const bool in = tok < p.M && col < p.K;
            if (!staged && in && p.accumulate) {
              const uint4 o0 = *reinterpret_cast<const uint4*>(d), o1 = *reinterpret_cast<const uint4*>(d + 8);
              const uint32_t ow[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                f[2 * j] += __uint_as_float(ow[j] << 16);
                f[2 * j + 1] += __uint_as_float(ow[j] & 0xffff0000u);
              }
            }
            uint32_t w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) w[j] = pack_bf16x2_rn(f[2 * j], f[2 * j + 1]);
            if (staged) {
              const uint32_t box = stg + (a * 4 + (c >> 6)) * 16384;
              const uint32_t ch = (c & 63) >> 3;
              sts_v4(box + sw128_offset(tr, ch), w[0], w[1], w[2], w[3]);
              sts_v4(box + sw128_offset(tr, ch + 1), w[4], w[5], w[6], w[7]);
            } else if (in) {
              *reinterpret_cast<uint4*>(d) = make_uint4(w[0], w[1], w[2], w[3]);
              *reinterpret_cast<uint4*>(d + 8) = make_uint4(w[4], w[5], w[6], w[7]);
            }
          }
        }
      }
    }
    if (staged) {
      fence_proxy_async_smem();
      named_bar_sync(1, kPrTeams * 128);
      if (threadIdx.x == 64 && ok) {
        if (!BWD) {
          for (int b = 0; b < 4; ++b)
            tma_store_2d(&tm_out, stg + b * 32768, pair * kPrCols + static_cast<int>(rank) * 128 + (b & 1) * 64,
                         tok0 + (b >> 1) * 256);
        } else {
          for (int b = 0; b < 8; ++b)
            tma_store_2d(&tm_out, stg + b * 16384, pair * kPrCols + (b & 3) * 64,
                         tok0 + (b >> 2) * 256 + static_cast<int>(rank) * 128);
        }
        tma_store_commit_and_wait_read();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA frees TMEM or leaves while the pair's MMAs may touch it
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tbase, 512);
  }
}

// Cluster of two along x, programmatic stream serialization.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pair(void (*kernel)(KArgs...), dim3 grid, cudaStream_t s, Args&&... args) {
  cudaError_t e = set_smem_limit_once(kernel, kPrSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kPrThreads);
  cfg.dynamicSmemBytes = kPrSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool use_pair_gemm(int M) { return M > 256; }

int fwd_pair_ctas(int M, int N) { return 2 * ((N + kPrCols - 1) / kPrCols) * ((M + kPrTokens - 1) / kPrTokens); }
int bwd_pair_ctas(int M, int K) { return 2 * ((K + kPrCols - 1) / kPrCols) * ((M + kPrTokens - 1) / kPrTokens); }

static PairParams pair_params(const Nf4Dev& w, const __nv_bfloat16* lora_b, const __nv_bfloat16* lora_a,
                              __nv_bfloat16* out, unsigned* status, int M, int r, int accumulate, uint64_t wait_ns) {
  PairParams prm;
  prm.codes = w.codes;
  prm.absq = w.absq;
  prm.step = w.step;
  prm.mean = w.mean;
  prm.lora_b = lora_b;
  prm.lora_a = lora_a;
  prm.out = out;
  prm.status = status;
  prm.M = M;
  prm.N = static_cast<int>(w.n);
  prm.K = static_cast<int>(w.k);
  prm.r = r;
  prm.lora_blocks = (r + 63) / 64;
  prm.accumulate = accumulate;
  prm.staged_store = 0;
  prm.wait_ns = wait_ns;
  return prm;
}

cudaError_t launch_fwd_gemm_pair(const __nv_bfloat16* x, int M, const Nf4Dev& w, const __nv_bfloat16* st,
                                 const __nv_bfloat16* lora_b, int r, __nv_bfloat16* y, unsigned* status,
                                 uint64_t wait_ns, cudaStream_t s) {
  const int N = static_cast<int>(w.n), K = static_cast<int>(w.k);
  CUtensorMap tx, tst;
  if (!make_tensor_map_bf16_2d(&tx, x, K, M, static_cast<uint64_t>(K) * 2, 64, 128)) return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tst, st, r, M, static_cast<uint64_t>(r) * 2, 64, 128)) return cudaErrorInvalidValue;
  PairParams prm = pair_params(w, lora_b, nullptr, y, status, M, r, 0, wait_ns);
  CUtensorMap ty = tst;
  prm.staged_store = (N % 8 == 0) && make_tensor_map_bf16_2d(&ty, y, N, M, static_cast<uint64_t>(N) * 2, 64, 256);
  const dim3 grid(2 * ((N + kPrCols - 1) / kPrCols), (M + kPrTokens - 1) / kPrTokens);
  return launch_pair(k_qgemm_pair<false>, grid, s, tx, tst, ty, prm);
}

cudaError_t launch_bwd_gemm_pair(const __nv_bfloat16* dy, int M, const Nf4Dev& w, const __nv_bfloat16* su,
                                 const __nv_bfloat16* lora_a, int r, __nv_bfloat16* dx, int accumulate,
                                 unsigned* status, uint64_t wait_ns, cudaStream_t s) {
  const int N = static_cast<int>(w.n), K = static_cast<int>(w.k);
  CUtensorMap tdy, tsu;
  if (!make_tensor_map_bf16_2d(&tdy, dy, N, M, static_cast<uint64_t>(N) * 2, 64, 128)) return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tsu, su, r, M, static_cast<uint64_t>(r) * 2, 64, 128)) return cudaErrorInvalidValue;
  PairParams prm = pair_params(w, nullptr, lora_a, dx, status, M, r, accumulate, wait_ns);
  CUtensorMap tdx = tsu;
  prm.staged_store = !accumulate && make_tensor_map_bf16_2d(&tdx, dx, K, M, static_cast<uint64_t>(K) * 2, 64, 128);
  const dim3 grid(2 * ((K + kPrCols - 1) / kPrCols), (M + kPrTokens - 1) / kPrTokens);
  return launch_pair(k_qgemm_pair<true>, grid, s, tdy, tsu, tdx, prm);
}

}  // namespace qlora
