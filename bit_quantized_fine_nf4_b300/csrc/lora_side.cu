// LoRA down-projections beside the CTA-pair GEMMs, on few SMs (Day 25 notes
// "Fine-tuning and LoRA/QLoRA", section 2.1: the branch B (A x); section 6.2:
// scaled by s = alpha / r): the forward's T = X A^T (t_save = T in fp32,
// sT = bf16(s T)) and the backward's U = dY B (sU = bf16(s U), B given as its
// k-major copy B^T [r, N]).
//
// Each CTA walks 128-token tiles: TMA streams X [128 tok x 64 k] and A_lora
// [RP x 64 k] (K-major, 128B swizzle; RP = r rounded up to 16, rows past r are
// zero) through a deep ring (an SM's read rate grows with the bytes in flight),
// one thread issues M = 128 x N = RP MMAs into a double-buffered TMEM
// accumulator, and four warps write t_save [M, r] and sT [M, lora_ld(r)].  The GEMM that consumes sT
// starts beside this kernel and waits for it only before its LoRA k block.
#include "common.cuh"
#include "kernels.h"

namespace qlora {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct SideParams {
  float* t_out;          // t_save [M, r] (or null)
  __nv_bfloat16* s_out;  // sT [M, lora_ld(r)]
  unsigned* status;
  int M, K, r, rp;
  int stages, stage_bytes;
  float scale;
  float t_scale;         // t_save = t_scale * (X A^T); 1 without dropout (1 / (1 - p) with it)
  // split k: work unit u = (tile u / splits, k blocks [(u % splits) kbps, + kbps)); splits > 1 adds
  // the units' float32 partials [split][tile][RP / 4][128] float4 in split order in the tile's last CTA
  int splits, kbps;
  float* partial;
  unsigned* counters;    // [tiles], zero before the launch; the last CTA of a tile resets its word
  unsigned long long wait_ns;
};
constexpr int kSideMaxSplits = 8;

constexpr int kSideThreads = 192;  // warp 0 TMA + TMEM, warp 1 MMA, warps 2..5 epilogue
constexpr int kSideMaxStages = 8;
constexpr int kSideBox = 128 * 128;  // [128 rows x 64] bf16

__global__ void __launch_bounds__(kSideThreads, 1)
    k_lora_side(const __grid_constant__ CUtensorMap tm_a,  // X [M, K]        box 64 x 128
                const __grid_constant__ CUtensorMap tm_b,  // A_lora [r, K]   box 64 x RP
                const SideParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = p.stages, SB = p.stage_bytes, RP = p.rp;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * SB);
  uint64_t* empty = full + kSideMaxStages;
  uint64_t* acc_full = empty + kSideMaxStages;  // [2]
  uint64_t* acc_empty = acc_full + 2;           // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  volatile int* vabort = abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = (p.M + 127) / 128;
  const int n1 = p.K / 64;
  const int units = tiles * p.splits;
  int* last_flag = abort_flag + 1;
  const uint32_t alloc = 2 * RP <= 32 ? 32 : 2 * RP <= 64 ? 64 : 128;
  const uint32_t idesc = idesc_bf16_f32(128, RP, 0, 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSideMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 128);
    }
    *abort_flag = 0;
    *last_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0) {
    __syncwarp();
    tmem_alloc(tmem_holder, alloc);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;
  // launched early (programmatic dependent launch): the set-up above overlaps the preceding kernel;
  // its input rows and the outputs may belong to the preceding kernels of the stream
  griddep_wait();
  // the GEMM that follows needs sT / sU only for its last k block; it may start now, since every
  // kernel before this one has completed
  griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      int g = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int tile = u / p.splits, kb0 = (u % p.splits) * p.kbps, kb1 = min(n1, kb0 + p.kbps);
        for (int i = kb0; i < kb1; ++i, ++g) {
          const int s = g % S;
          if (!mbar_wait(&empty[s], ((g / S) & 1) ^ 1, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); ok = false; break; }
          uint8_t* st = smem + s * SB;
          mbar_arrive_expect_tx(&full[s], kSideBox + RP * 128);
          tma_load_2d(st, &tm_a, &full[s], i * 64, tile * 128);
          tma_load_2d(st + kSideBox, &tm_b, &full[s], i * 64, 0);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int g = 0, j = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++j) {
        const int kb0 = (u % p.splits) * p.kbps, kb1 = min(n1, kb0 + p.kbps);
        const int buf = j & 1;
        if (!mbar_wait(&acc_empty[buf], ((j >> 1) & 1) ^ 1, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); break; }
        tc_fence_after();
        const uint32_t d = tbase + buf * RP;
        for (int i = kb0; i < kb1; ++i, ++g) {
          const int s = g % S;
          if (!mbar_wait(&full[s], (g / S) & 1, p.wait_ns, vabort)) { abort_cta(p.status, abort_flag); ok = false; break; }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + s * SB);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ss(d, sdesc_sw128(a + kk * 32, 16, 1024), sdesc_sw128(a + kSideBox + kk * 32, 16, 1024), idesc,
                        (i > kb0 || kk > 0) ? 1u : 0u);
          mma_commit(&empty[s]);
        }
        if (ok) mma_commit(&acc_full[buf]);
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (128 threads)
    const int quarter = warp & 3;          // this warp's TMEM lane quarter
    const int lrow = quarter * 32 + lane;  // TMEM lane = token row of the tile
    const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
    int j = 0;
    const int rk = lora_ld(p.r);  // sT row stride; columns r .. rk-1 are zero (A rows past r load as zero)
    // t_save and sT of 4 consecutive columns c .. c + 3 of row tok from their float32 sums
    auto store4 = [&](int tok, int c, const float (&acc)[4]) {
      const float f[4] = {__fmul_rn(acc[0], p.t_scale), __fmul_rn(acc[1], p.t_scale), __fmul_rn(acc[2], p.t_scale),
                          __fmul_rn(acc[3], p.t_scale)};
      if (c < rk)  // rk % 8 == 0: four consecutive columns are all inside rk or all past it
        *reinterpret_cast<uint2*>(p.s_out + static_cast<int64_t>(tok) * rk + c) =
            make_uint2(pack_bf16x2_rn(__fmul_rn(f[0], p.scale), __fmul_rn(f[1], p.scale)),
                       pack_bf16x2_rn(__fmul_rn(f[2], p.scale), __fmul_rn(f[3], p.scale)));
      if (p.t_out == nullptr) return;
      float* to = p.t_out + static_cast<int64_t>(tok) * p.r + c;
      if ((p.r & 3) == 0) {  // rows of t_save start on 16-byte boundaries
        if (c < p.r) *reinterpret_cast<float4*>(to) = make_float4(f[0], f[1], f[2], f[3]);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c + e < p.r) to[e] = f[e];
      }
    };
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
      const int tile = u / p.splits, sp = u % p.splits;
      const int buf = j & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (j >> 1) & 1, p.wait_ns, vabort));
      if (!ok) break;
      tc_fence_after();
      const int tok = tile * 128 + lrow;
      if (p.splits > 1) {
        // this unit's partial: [RP / 4 column groups][128 rows] float4 (a warp stores 512 contiguous bytes)
        float4* part = reinterpret_cast<float4*>(p.partial) +
                       (static_cast<int64_t>(sp) * tiles + tile) * (RP / 4) * 128 + lrow;
        for (int c = 0; c < RP; c += 16) {
          uint32_t v[16];
          __syncwarp();
          tmem_ld_32x32b_x16(tbase + lane_field + buf * RP + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int q = 0; q < 16; q += 4)
            part[((c + q) >> 2) * 128] = make_float4(__uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                                     __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
        __threadfence();
        named_bar_sync(1, 128);
        if (lrow == 0) *last_flag = atomicAdd(p.counters + tile, 1u) == static_cast<unsigned>(p.splits - 1);
        named_bar_sync(1, 128);
        if (*reinterpret_cast<volatile int*>(last_flag)) {
          // the tile's last unit: every split's loads of one (column group, row) item, then their sum in split order
          __threadfence();
          const float4* src = reinterpret_cast<const float4*>(p.partial) + static_cast<int64_t>(tile) * (RP / 4) * 128;
          const int64_t sstride = static_cast<int64_t>(tiles) * (RP / 4) * 128;
          for (int c4 = 0; c4 < RP / 4; ++c4) {
            float4 v[kSideMaxSplits];
#pragma unroll
            for (int e = 0; e < kSideMaxSplits; ++e)
              v[e] = e < p.splits ? __ldcg(src + e * sstride + c4 * 128 + lrow) : make_float4(0.f, 0.f, 0.f, 0.f);
            float acc[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
            for (int e = 1; e < kSideMaxSplits; ++e) {
              if (e < p.splits) {
                acc[0] += v[e].x;
                acc[1] += v[e].y;
                acc[2] += v[e].z;
                acc[3] += v[e].w;
              }
            }
            if (tok < p.M) store4(tok, 4 * c4, acc);
          }
          if (lrow == 0) p.counters[tile] = 0u;
        }
        continue;
      }
      for (int c = 0; c < RP; c += 16) {
        uint32_t v[16];
        __syncwarp();
        tmem_ld_32x32b_x16(tbase + lane_field + buf * RP + c, v);
        tmem_ld_wait();
        if (tok < p.M) {
#pragma unroll
          for (int q = 0; q < 16; q += 4) {
            const float acc[4] = {__uint_as_float(v[q]), __uint_as_float(v[q + 1]), __uint_as_float(v[q + 2]),
                                  __uint_as_float(v[q + 3])};
            store4(tok, c + q, acc);
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
    tmem_dealloc(tbase, alloc);
  }
}

// ------------------------------------------------------------------ host
bool lora_side_supported(int r) { return r >= 1 && r <= 64; }

// U = dY B: k split so the units fill the GPU (at most kSideMaxSplits per 128-row tile).
static void side_split(int M, int K, int num_sms, int* splits, int* kbps) {
  const int tiles = (M + 127) / 128, n1 = K / 64;
  int sp = num_sms / (tiles > 0 ? tiles : 1);
  if (sp > kSideMaxSplits) sp = kSideMaxSplits;
  if (sp > n1) sp = n1;
  if (sp < 1) sp = 1;
  *kbps = (n1 + sp - 1) / sp;
  *splits = (n1 + *kbps - 1) / *kbps;
}

size_t lora_side_bwd_workspace_bytes(int M, int K, int r, int num_sms) {
  int splits = 1, kbps = 1;
  side_split(M, K, num_sms, &splits, &kbps);
  if (splits == 1) return 0;
  const size_t tiles = (M + 127) / 128, rp = (r + 15) / 16 * 16;
  return align_up(splits * tiles * 128 * rp * 4, 256) + align_up(tiles * 4, 256);
}

static cudaError_t launch_side(const __nv_bfloat16* in, const __nv_bfloat16* mt, int M, int K, int r, float scale,
                               float* t_out, __nv_bfloat16* s_out, int max_ctas, int splits, int kbps, float* partial,
                               unsigned* counters, unsigned* status, uint64_t wait_ns, cudaStream_t s, float t_scale) {
  const int rp = (r + 15) / 16 * 16;
  CUtensorMap ta, tb;
  if (!make_tensor_map_bf16_2d(&ta, in, K, M, static_cast<uint64_t>(K) * 2, 64, 128)) return cudaErrorInvalidValue;
  if (!make_tensor_map_bf16_2d(&tb, mt, K, r, static_cast<uint64_t>(K) * 2, 64, rp)) return cudaErrorInvalidValue;
  SideParams prm = {};
  prm.t_out = t_out;
  prm.s_out = s_out;
  prm.status = status;
  prm.M = M;
  prm.K = K;
  prm.r = r;
  prm.rp = rp;
  prm.stage_bytes = kSideBox + rp * 128;
  prm.stages = (200 * 1024) / prm.stage_bytes;
  if (prm.stages > kSideMaxStages) prm.stages = kSideMaxStages;
  prm.scale = scale;
  prm.t_scale = t_scale;
  prm.splits = splits;
  prm.kbps = kbps;
  prm.partial = partial;
  prm.counters = counters;
  prm.wait_ns = wait_ns;
  const size_t smem = 1024 + static_cast<size_t>(prm.stages) * prm.stage_bytes + (2 * kSideMaxStages + 4) * 8 + 16;
  const int units = (M + 127) / 128 * splits;
  int grid = units < max_ctas ? units : max_ctas;
  if (grid >= 2) grid &= ~1;  // clusters of two: whole TPCs stay free for the pair GEMM
  if (grid < 1) grid = 1;
  cudaError_t e = set_smem_limit_once(k_lora_side, 232448);  // once per kernel: the largest size any rank needs
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSideThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = grid >= 2 ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, k_lora_side, ta, tb, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_lora_side_fwd(const __nv_bfloat16* x, const __nv_bfloat16* lora_a, int M, int K, int r, float scale,
                                 float* t_save, __nv_bfloat16* st, int max_ctas, unsigned* status, uint64_t wait_ns,
                                 cudaStream_t s, float t_scale) {
  return launch_side(x, lora_a, M, K, r, scale, t_save, st, max_ctas, 1, K / 64, nullptr, nullptr, status, wait_ns, s,
                     t_scale);
}

cudaError_t launch_lora_side_bwd(const __nv_bfloat16* dy, const __nv_bfloat16* bt, int M, int N, int r, float scale,
                                 __nv_bfloat16* su, void* ws, int num_sms, unsigned* status, uint64_t wait_ns,
                                 cudaStream_t s) {
  int splits = 1, kbps = 1;
  side_split(M, N, num_sms, &splits, &kbps);
  float* partial = nullptr;
  unsigned* counters = nullptr;
  if (splits > 1) {
    const size_t tiles = (M + 127) / 128, rp = (r + 15) / 16 * 16;
    partial = static_cast<float*>(ws);
    counters = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + align_up(splits * tiles * 128 * rp * 4, 256));
  }
  return launch_side(dy, bt, M, N, r, scale, nullptr, su, num_sms, splits, kbps, partial, counters, status, wait_ns, s,
                     1.0f);
}

unsigned* lora_side_bwd_counters(void* ws, int M, int K, int r, int num_sms) {
  int splits = 1, kbps = 1;
  side_split(M, K, num_sms, &splits, &kbps);
  if (splits == 1) return nullptr;
  const size_t tiles = (M + 127) / 128, rp = (r + 15) / 16 * 16;
  return reinterpret_cast<unsigned*>(static_cast<char*>(ws) + align_up(splits * tiles * 128 * rp * 4, 256));
}

}  // namespace qlora
