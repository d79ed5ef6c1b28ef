// NF4 QLoRA GEMMs on CTA pairs (tcgen05 cta_group::2), for token counts > 256.
//
// The frozen product of the QLoRA linear (glossary "QLoRA", "How QLoRA works":
// the NF4 weight is dequantised to bfloat16 for the matmul, the LoRA output is
// added; Day 25 notes "Fine-tuning and LoRA/QLoRA", section 2.1, scaled by
// s = alpha / r as in section 6.2).  Both directions compute D[tokens, columns]:
//
//   forward   Y[m, n]  = sum_k X[m, k] deq(W)[n, k]   + sum_j sT[m, j] B[n, j]
//   backward  dX[m, k] = sum_n dY[m, n] deq(W)[n, k]  + sum_j sU[m, j] A[j, k]
//
// A operand = activation rows (tokens) by TMA; B operand = this CTA's half of
// the pair's 256 output columns of deq(W), decoded by the producer warps
// (forward: K-major W rows; backward: MN-major, 64 n rows x 128 columns).
// The dequantisation runs on the ALU pipe (about four integer ops per weight),
// so a decoded weight has to feed enough MMA work: the pair decodes a 64 x 256
// slice of W per k step and uses it for 512 tokens (two M = 256 x N = 256
// accumulators, 512 TMEM columns per CTA).  Per SM and k step: 32 KB of TMA
// fills, 16 KB of decoded W, 8 MMAs (1024 tensor cycles).
//
// Roles per CTA (576 threads): warp 0 lane 0 = TMA, warp 0 = TMEM allocation;
// warp 1 lane 0 of the even CTA = MMA issue; warps 2..17 = four producer teams
// (k steps round-robin) that decode one W slice each into shared memory (or
// copy the LoRA rows for the last k steps), then the epilogue.
//
// Stage (48 KB): [0, 32K) two TMA boxes [128 tokens x 64] bf16 (one per
// accumulator), K-major 128B swizzle; [32K, 48K) the decoded W tile.
// "Stage s full" is one barrier in the even CTA that both CTAs complete: the odd
// CTA's TMA signals it across the pair and its producer warps arrive remotely,
// so the MMA thread waits once per k step.  "Stage s empty" lives in both CTAs
// and is released by one multicast MMA commit.  The result is staged in the
// freed stage buffers and written with TMA stores.
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
  int out_cols;                 // forward N, backward K
  int lora_blocks, accumulate;
  int staged_store;             // write the result through shared memory with TMA stores (tm_out)
  unsigned long long wait_ns;
};

constexpr int kPrTeams = 4;
constexpr int kPrThreads = 64 + kPrTeams * 128;
constexpr int kPrStages = kPrTeams;                 // team t always fills stage t
constexpr uint32_t kPrBox = 128 * 128;              // [128 tokens x 64] bf16
constexpr uint32_t kPrActBytes = 2 * kPrBox;        // one box per accumulator
constexpr uint32_t kPrProdBytes = 16384;            // decoded W tile of this CTA
constexpr uint32_t kPrStage = kPrActBytes + kPrProdBytes;
constexpr uint32_t kPrBarBase = kPrStages * kPrStage;
constexpr int kPrBars = 2 * kPrStages + 1;
constexpr size_t kPrSmem = 1024 + kPrBarBase + kPrBars * 8 + 16;
static_assert(kPrSmem <= 232448, "dynamic shared memory per block");
constexpr int kPrTokens = 512;  // tokens per pair tile
constexpr int kPrCols = 256;    // output columns per pair tile (W rows forward, W columns backward)

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
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1)
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
  // accumulator a holds tokens tok0 + 256 a + [0, 256); this CTA supplies the
  // A rows (and holds the D rows) 128 rank + [0, 128) of each
  const int ta = tok0 + static_cast<int>(rank) * 128, tb = ta + 256;
  const int cta_col0 = pair * kPrCols + static_cast<int>(rank) * 128;  // first of this CTA's 128 B columns

  // producer unit of this thread (warps 2..17); its first codes are fetched before the set-up
  const int team = (warp - 2) >> 2;
  const int t = ((warp - 2) & 3) * 32 + lane;  // 0..127
  const float mu = *p.mean;
  const int kb_row = p.K / 64;
  // forward: W row n_fix, k block i;  backward: W row i * 64 + rrow, k block kblk (columns col0 .. + 63)
  const int n_fix = cta_col0 + t;
  const uint32_t rrow = t & 63, slab = t >> 6;
  const int col0 = cta_col0 + static_cast<int>(slab) * 64;
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
  if (threadIdx.x == 32) {
    // warm L2 with the first activation boxes while the pair sets up
    for (int i = 0; i < kPrStages && i < n_main; ++i) {
      if (ta < p.M) tma_prefetch_l2_2d(&tm_act, i * 64, ta);
      if (tb < p.M) tma_prefetch_l2_2d(&tm_act, i * 64, tb);
    }
  }

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
        // no LoRA k steps: still wait for the preceding kernel, before the last stage so that the
        // epilogue (which lets the next kernel launch) runs only after the wait has returned
        if (p.lora_blocks == 0 && i == n_iter - 1) griddep_wait();
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
      griddep_wait();  // returns at once after the waits above; covers a loop ended by an abort
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
          const uint64_t bd = BWD ? sdesc_sw128(prod + kk * 2048, 8192, 1024) : sdesc_sw128(prod + kk * 32, 16, 1024);
#pragma unroll
          for (int a = 0; a < 2; ++a)
            mma_pair_bf16_ss(tbase + a * 256, sdesc_sw128(act + a * kPrBox + kk * 32, 16, 1024), bd, idesc,
                             (i > 0 || kk > 0) ? 1u : 0u);
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
      const int s = i % kPrStages;
      const uint32_t ph = (i / kPrStages) & 1;
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
        // LoRA B: K-major row n_fix, 64 j
        load_lora_b_row(p.lora_b, n_fix, p.N, p.r, (i - n_main) * 64, words);
      } else {
        // LoRA A: MN-major row j = jb + rrow, 64 output columns from col0
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
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&empty[s], ph ^ 1, p.wait_ns, vabort));
      if (!ok) { if (lane == 0) abort_cta(p.status, abort_flag); alive = false; break; }
      const uint32_t base = smem_u32(smem + s * kPrStage + kPrActBytes);
      // forward: row t of a [128 x 64] K-major tile; backward: row rrow of 64-column slab `slab`
      const uint32_t rbase = BWD ? base + slab * 8192 : base;
      const uint32_t row = BWD ? rrow : static_cast<uint32_t>(t);
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        sts_v4(rbase + sw128_offset(row, ch), words[4 * ch], words[4 * ch + 1], words[4 * ch + 2], words[4 * ch + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&full[s]);
        else
          mbar_arrive_cluster_addr(full_remote);
      }
    }
    // ---------------------------------------------------------------- epilogue
    bool ok = __all_sync(0xffffffffu, mbar_wait(acc_full, 0, p.wait_ns, vabort));
    ok = __all_sync(0xffffffffu, ok && !*vabort);
    tc_fence_after();
    // this CTA's loads of the preceding kernels' outputs are done: the next kernel may launch
    griddep_launch_dependents();
    const int quarter = warp & 3;    // TMEM lanes 32 quarter .. + 31
    const int wq = (warp - 2) >> 2;  // 0..3 among the warps of this lane quarter: columns 64 wq .. + 63
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    const bool staged = p.staged_store && !p.accumulate;
    // staged: 8 boxes [128 tokens x 64 columns], box (accumulator a, column slab wq), 128B swizzle
    const uint32_t stg = smem_u32(smem);
    const uint32_t tr = quarter * 32 + lane;
    if (ok) {
      for (int a = 0; a < 2; ++a) {
        uint32_t v[64];
        uint32_t(&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(v);
        uint32_t(&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(v + 32);
        __syncwarp();
        tmem_ld_32x32b_x32(tbase + lane_field + a * 256 + wq * 64, v0);
        tmem_ld_32x32b_x32(tbase + lane_field + a * 256 + wq * 64 + 32, v1);
        tmem_ld_wait();
        const int tok = tok0 + a * 256 + static_cast<int>(rank) * 128 + static_cast<int>(tr);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {  // 8 columns per 16-byte chunk
          float f[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(v[ch * 8 + j]);
          const int col = pair * kPrCols + wq * 64 + ch * 8;
          if (staged) {
            sts_v4(stg + (a * 4 + wq) * 16384 + sw128_offset(tr, ch), pack_bf16x2_rn(f[0], f[1]),
                   pack_bf16x2_rn(f[2], f[3]), pack_bf16x2_rn(f[4], f[5]), pack_bf16x2_rn(f[6], f[7]));
          } else if (tok < p.M) {
            __nv_bfloat16* d = p.out + static_cast<int64_t>(tok) * p.out_cols + col;
            if ((p.out_cols & 7) == 0 && col + 8 <= p.out_cols) {
              // 16-byte read-modify-write (accumulate: float32 sum of the old bf16 and the result)
              uint4* d4 = reinterpret_cast<uint4*>(d);
              if (p.accumulate) {
                const uint4 o = *d4;
                const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  f[2 * j] += __uint_as_float(ow[j] << 16);
                  f[2 * j + 1] += __uint_as_float(ow[j] & 0xffff0000u);
                }
              }
              *d4 = make_uint4(pack_bf16x2_rn(f[0], f[1]), pack_bf16x2_rn(f[2], f[3]), pack_bf16x2_rn(f[4], f[5]),
                               pack_bf16x2_rn(f[6], f[7]));
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                if (col + j < p.out_cols) {
                  const float o = p.accumulate ? __bfloat162float(d[j]) : 0.f;
                  d[j] = __float2bfloat16_rn(f[j] + o);
                }
              }
            }
          }
        }
      }
    }
    if (staged) {
      fence_proxy_async_smem();
      named_bar_sync(1, kPrTeams * 128);
      if (threadIdx.x == 64 && ok) {
        for (int b = 0; b < 8; ++b)
          tma_store_2d(&tm_out, stg + b * 16384, pair * kPrCols + (b & 3) * 64,
                       tok0 + (b >> 2) * 256 + static_cast<int>(rank) * 128);
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
  prm.out_cols = 0;
  prm.staged_store = 0;
  prm.wait_ns = wait_ns;
  return prm;
}

cudaError_t launch_fwd_gemm_pair(const __nv_bfloat16* x, int M, const Nf4Dev& w, const __nv_bfloat16* st,
                                 const __nv_bfloat16* lora_b, int r, __nv_bfloat16* y, unsigned* status,
                                 uint64_t wait_ns, cudaStream_t s) {
  const int N = static_cast<int>(w.n), K = static_cast<int>(w.k);
  CUtensorMap tx, tst;
  const int rk = lora_ld(r);
  if (!make_tensor_map_bf16_2d(&tx, x, K, M, static_cast<uint64_t>(K) * 2, 64, 128)) return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tst, st, rk, M, static_cast<uint64_t>(rk) * 2, 64, 128)) return cudaErrorInvalidValue;
  PairParams prm = pair_params(w, lora_b, nullptr, y, status, M, r, 0, wait_ns);
  prm.out_cols = N;
  CUtensorMap ty = tst;
  prm.staged_store = (N % 8 == 0) && make_tensor_map_bf16_2d(&ty, y, N, M, static_cast<uint64_t>(N) * 2, 64, 128);
  const dim3 grid(2 * ((N + kPrCols - 1) / kPrCols), (M + kPrTokens - 1) / kPrTokens);
  return launch_pair(k_qgemm_pair<false>, grid, s, tx, tst, ty, prm);
}

cudaError_t launch_bwd_gemm_pair(const __nv_bfloat16* dy, int M, const Nf4Dev& w, const __nv_bfloat16* su,
                                 const __nv_bfloat16* lora_a, int r, __nv_bfloat16* dx, int accumulate,
                                 unsigned* status, uint64_t wait_ns, cudaStream_t s, int with_lora) {
  const int N = static_cast<int>(w.n), K = static_cast<int>(w.k);
  CUtensorMap tdy, tsu;
  const int rk = lora_ld(r);
  if (!make_tensor_map_bf16_2d(&tdy, dy, N, M, static_cast<uint64_t>(N) * 2, 64, 128)) return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tsu, su, rk, M, static_cast<uint64_t>(rk) * 2, 64, 128)) return cudaErrorInvalidValue;
  PairParams prm = pair_params(w, nullptr, lora_a, dx, status, M, r, accumulate, wait_ns);
  if (!with_lora) prm.lora_blocks = 0;
  prm.out_cols = K;
  CUtensorMap tdx = tsu;
  prm.staged_store = !accumulate && make_tensor_map_bf16_2d(&tdx, dx, K, M, static_cast<uint64_t>(K) * 2, 64, 128);
  const dim3 grid(2 * ((K + kPrCols - 1) / kPrCols), (M + kPrTokens - 1) / kPrTokens);
  return launch_pair(k_qgemm_pair<true>, grid, s, tdy, tsu, tdx, prm);
}

}  // namespace qlora
