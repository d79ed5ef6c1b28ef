// NF4 quantisation, double quantisation of the block scales, and dequantisation.
//
// Ultralytics glossary "QLoRA", section "How QLoRA works": one absmax scale per
// block of 64 weights, 4-bit code = index of the NF4 level nearest to
// w / absmax, restored weight = level * scale; the block scales are quantised
// again to 8 bits in groups of 256.  fedte.cc "QLoRA fine-tuning on 4 GB",
// section 1: two codes per byte (0.5 byte per parameter).
//
// Layout in HBM (row-major weight [n, k], k % 64 == 0):
//   codes       uint8 [n*k/2]    element 2i in the high nibble of byte i
//   absmax_q    int8  [n*k/64]   double-quantised block scales
//   absmax_step f32   [ceil(n*k/64/256)]
//   absmax_mean f32   [1]
//
// Bit-exactness: every float32 operation that decides a code or a dequantised
// value is an explicitly rounded intrinsic (__fdiv_rn / __fsub_rn / __fmul_rn /
// __fadd_rn / rintf / bf16 round-to-nearest), so no FMA contraction changes it.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace qlora {

// ------------------------------------------------------------------ encode thresholds
// Monotone integer key of a float (total order of non-NaN floats, -0 == +0).
__device__ __forceinline__ int32_t f32_key(float f) {
  const int32_t b = __float_as_int(f);
  return b >= 0 ? b : -(b & 0x7fffffff);
}
__device__ __forceinline__ float key_f32(int32_t k) {
  return k >= 0 ? __int_as_float(k) : __int_as_float((-k) | static_cast<int32_t>(0x80000000u));
}

// Threshold t_j (j = 0..14): the smallest float x with |x - L[j+1]| < |x - L[j]|
// in float32 arithmetic.  For x between the two levels both distances are
// monotone in x, so "x is strictly nearer to L[j+1]" switches exactly once and
// a bisection over the ordered floats finds the switch.  Then the nearest
// level with ties to the lower index is code(x) = #{ j : x >= t_j }.
__device__ float nf4_threshold(int j) {
  const float lo = nf4_level(j), hi = nf4_level(j + 1);
  int32_t a = f32_key(lo), b = f32_key(hi);  // predicate false at a, true at b
  while (b - a > 1) {
    const int32_t mid = a + (b - a) / 2;
    const float x = key_f32(mid);
    const bool nearer_hi = __fsub_rn(hi, x) < __fsub_rn(x, lo);
    if (nearer_hi) b = mid; else a = mid;
  }
  return key_f32(b);
}

struct Thresholds {
  float t[15];
};

__device__ __forceinline__ uint32_t nf4_code(const Thresholds& th, float x) {
  const bool b3 = x >= th.t[7];
  const bool b2 = x >= (b3 ? th.t[11] : th.t[3]);
  const float m1 = b3 ? (b2 ? th.t[13] : th.t[9]) : (b2 ? th.t[5] : th.t[1]);
  const bool b1 = x >= m1;
  const float m0 = b3 ? (b2 ? (b1 ? th.t[14] : th.t[12]) : (b1 ? th.t[10] : th.t[8]))
                      : (b2 ? (b1 ? th.t[6] : th.t[4]) : (b1 ? th.t[2] : th.t[0]));
  const bool b0 = x >= m0;
  return (b3 ? 8u : 0u) | (b2 ? 4u : 0u) | (b1 ? 2u : 0u) | (b0 ? 1u : 0u);
}

// ------------------------------------------------------------------ quantise
template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[8]) {
  const uint4 a = ldg_nc_v4(p), b = ldg_nc_v4(p + 4);
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y); v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y); v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 a = ldg_nc_v4(p);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// Each thread quantises 8 consecutive elements; 8 lanes share one 64-block.
template <typename T>
__global__ void __launch_bounds__(256) k_nf4_quantize(const T* __restrict__ w, int64_t n_elems,
                                                      uint8_t* __restrict__ codes, float* __restrict__ absmax,
                                                      unsigned* status) {
  __shared__ float s_thr[16];
  if (threadIdx.x < 15) s_thr[threadIdx.x] = nf4_threshold(threadIdx.x);
  __syncthreads();
  Thresholds th;
#pragma unroll
  for (int j = 0; j < 15; ++j) th.t[j] = s_thr[j];

  const int lane = threadIdx.x & 31;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t n_tiles = (n_elems + 255) >> 8;
  for (int64_t tile = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); tile < n_tiles;
       tile += warps_total) {
    const int64_t e0 = tile * 256 + lane * 8;
    const bool valid = e0 < n_elems;  // whole 64-blocks: e0 < n  =>  e0 + 8 <= n
    float v[8];
    if (valid) {
      load8<T>(w + e0, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    }
    uint32_t mb = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mb = max(mb, __float_as_uint(v[i]) & 0x7fffffffu);
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
    if (!valid) continue;
    if (mb >= 0x7f800000u && (lane & 7) == 0) latch_status(status, ST_NONFINITE);
    const float a = __uint_as_float(mb);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float x = (mb == 0) ? 0.f : __fdiv_rn(v[i], a);
      const uint32_t c = nf4_code(th, x);
      packed |= c << ((i >> 1) * 8 + ((i & 1) ? 0 : 4));
    }
    reinterpret_cast<uint32_t*>(codes)[e0 >> 3] = packed;
    if ((lane & 7) == 0) absmax[e0 >> 6] = a;
  }
}

// ------------------------------------------------------------------ exact mean of the absmax values
// The mean is float32( RN64(sum a_i) / n ) where RN64(sum) is the exactly
// rounded float64 value of the exact sum, so it does not depend on the order
// in which blocks are visited.  The exact sum is accumulated as integers: a
// float32 a = m * 2^(max(e,1) - 150) (m the 24-bit significand, e the biased
// exponent field), so sum_i a_i = sum_e B[e] * 2^(max(e,1) - 150) with
// B[e] = sum of m over values with exponent field e (64-bit, exact for up to
// 2^40 values).  The last CTA turns the bins into a 320-bit integer and
// rounds it once to float64 (round to nearest, ties to even).
__device__ double exact_bins_to_double(const unsigned long long* bins) {  // bins: shared memory
  uint64_t limb[6] = {0, 0, 0, 0, 0, 0};  // little-endian 384-bit accumulator of sum * 2^149
  for (int e = 0; e < 255; ++e) {
    const uint64_t v = bins[e];
    if (!v) continue;
    const int sh = (e < 1 ? 1 : e) - 1;  // 0..253
    const int li = sh >> 6, bo = sh & 63;
    const uint64_t lo = v << bo;
    const uint64_t hi = bo ? (v >> (64 - bo)) : 0;
    uint64_t old = limb[li];
    limb[li] = old + lo;
    uint64_t carry = limb[li] < old ? 1 : 0;
    for (int t = li + 1; t < 6; ++t) {
      const uint64_t add = (t == li + 1 ? hi : 0) + carry;  // hi < 2^46, no overflow
      old = limb[t];
      limb[t] = old + add;
      carry = limb[t] < old ? 1 : 0;
      if (!carry && t > li + 1) break;
    }
  }
  int top = -1;  // index of the most significant set bit
  for (int t = 5; t >= 0; --t)
    if (limb[t]) { top = t * 64 + 63 - __clzll(static_cast<long long>(limb[t])); break; }
  if (top < 0) return 0.0;
  auto bit = [&](int i) -> uint64_t { return (i < 0) ? 0 : ((limb[i >> 6] >> (i & 63)) & 1ull); };
  if (top <= 52) {
    uint64_t mant = limb[0];  // < 2^53, exact
    return ldexp(static_cast<double>(mant), -149);
  }
  const int shift = top - 52;  // keep bits [shift, top]
  uint64_t mant = 0;
  for (int i = top; i >= shift; --i) mant = (mant << 1) | bit(i);
  const uint64_t round = bit(shift - 1);
  uint64_t sticky = 0;
  for (int i = shift - 2; i >= 0 && !sticky; --i) sticky |= bit(i);
  int exp2 = shift - 149;
  if (round && (sticky || (mant & 1ull))) {
    mant += 1;
    if (mant == (1ull << 53)) { mant >>= 1; exp2 += 1; }
  }
  return ldexp(static_cast<double>(mant), exp2);
}

__global__ void __launch_bounds__(256) k_absmax_mean(const float* __restrict__ absmax, int64_t n_a,
                                                     unsigned long long* bins, unsigned* counter, float* mean_out,
                                                     unsigned* status) {
  __shared__ unsigned long long s_bins[256];
  __shared__ int s_last;
  for (int i = threadIdx.x; i < 256; i += blockDim.x) s_bins[i] = 0;
  __syncthreads();
  // whole warps walk the array; lanes holding the same exponent add their
  // mantissas in the warp (< 32 * 2^24, exact in 32 bits) and one of them adds
  // the group's sum to the shared bin
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < n_a; base += stride) {
    const int64_t i = base + threadIdx.x;
    uint32_t e = 256, m = 0;  // 256: no value in this lane
    if (i < n_a) {
      const uint32_t u = __float_as_uint(absmax[i]) & 0x7fffffffu;
      e = u >> 23;
      if (e >= 255) {
        latch_status(status, ST_NONFINITE);
        e = 256;
      } else {
        m = (e == 0) ? (u & 0x7fffffu) : ((u & 0x7fffffu) | 0x800000u);
      }
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const unsigned sum = __reduce_add_sync(grp, m);
    if (e < 255 && sum && (threadIdx.x & 31) == __ffs(grp) - 1)
      atomicAdd(&s_bins[e], static_cast<unsigned long long>(sum));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (s_bins[i]) atomicAdd(bins + i, s_bins[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counter, 1u) == gridDim.x - 1);
  __syncthreads();
  if (s_last) {
    // the last CTA reads all bins at once, then one thread converts them exactly
    __threadfence();
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s_bins[i] = __ldcg(bins + i);
    __syncthreads();
    if (threadIdx.x == 0) {
      const double s = exact_bins_to_double(s_bins);
      *mean_out = __double2float_rn(__ddiv_rn(s, static_cast<double>(n_a)));
    }
  }
}

// One CTA per group of 256 absmax values: step = max|a - mu| / 127,
// q = clamp(rint((a - mu) / step), -127, 127), q = 0 when step == 0.
__global__ void __launch_bounds__(256) k_absmax_dq(const float* __restrict__ absmax, int64_t n_a,
                                                   const float* __restrict__ mean, int8_t* __restrict__ q,
                                                   float* __restrict__ step) {
  __shared__ float s_max[8];
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  const bool valid = i < n_a;
  const float mu = *mean;
  const float d = valid ? __fsub_rn(absmax[i], mu) : 0.f;
  float m = fabsf(d);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = m;
  __syncthreads();
  m = s_max[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) m = fmaxf(m, s_max[w]);
  const float st = __fdiv_rn(m, 127.0f);
  if (threadIdx.x == 0) step[blockIdx.x] = st;
  if (!valid) return;
  int qi = 0;
  if (st != 0.f) {
    float r = rintf(__fdiv_rn(d, st));
    r = fminf(fmaxf(r, -127.f), 127.f);
    qi = static_cast<int>(r);
  }
  q[i] = static_cast<int8_t>(qi);
}

// ------------------------------------------------------------------ dequantise
// One thread per 64-block; each warp stages its 32 blocks (4 KB of bf16) in
// shared memory with a chunk swizzle and writes them out as 512-byte
// coalesced rows.
__global__ void __launch_bounds__(256) k_nf4_dequantize(const uint8_t* __restrict__ codes,
                                                        const int8_t* __restrict__ absq,
                                                        const float* __restrict__ step,
                                                        const float* __restrict__ mean,
                                                        uint16_t* __restrict__ out, int64_t n_blocks) {
  __shared__ uint4 s_out[8][256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float mu = *mean;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * 8;
  const int64_t n_tiles = (n_blocks + 31) >> 5;
  for (int64_t tile = static_cast<int64_t>(blockIdx.x) * 8 + warp; tile < n_tiles; tile += warps_total) {
    const int64_t b = tile * 32 + lane;
    uint32_t o[32];
    if (b < n_blocks) {
      const uint4 c0 = ldg_nc_v4(codes + b * 32), c1 = ldg_nc_v4(codes + b * 32 + 16);
      const float a2 = restore_absmax(absq[b], step[b >> 8], mu);
      nf4_decode_block(c0, c1, a2, o);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = 0;
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
      s_out[warp][lane * 8 + (c ^ (lane & 7))] = make_uint4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int idx = j * 32 + lane;
      const int row = idx >> 3, chunk = idx & 7;
      const int64_t bb = tile * 32 + row;
      if (bb < n_blocks)
        reinterpret_cast<uint4*>(out + bb * 64)[chunk] = s_out[warp][row * 8 + (chunk ^ (row & 7))];
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ fixed scratch (no-allocation entry point)
// Scratch of qlora_nf4_quantize_noalloc: the float32 absmax of up to
// kNoAllocMaxBlocks blocks of 64 weights, then the 256 exact-sum bins and the
// CTA counter of the mean.  It is module-scope device memory: every device
// that loads the library holds one copy until the process exits.  All calls
// on a device share it; the bins and the counter are cleared by every call,
// the absmax region is fully rewritten, so nothing carries over -- but two
// calls whose kernels overlap on the GPU race on it.
constexpr int64_t kNoAllocMaxBlocks = int64_t(1) << 20;  // n*k <= 2^26 weights
constexpr size_t kNoAllocBinsOffset = static_cast<size_t>(kNoAllocMaxBlocks) * 4;
constexpr size_t kNoAllocBytes = kNoAllocBinsOffset + 256 * 8 + 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

int64_t noalloc_max_weights() { return kNoAllocMaxBlocks * 64; }

// Device address of the scratch on the current device.  The first call on a
// device looks it up with cudaGetSymbolAddress (the host-side name of a
// __device__ array is not a device address) and caches it per device.
cudaError_t noalloc_scratch(float** absmax, void** bins) {
  static std::mutex mu;
  static void* addr[128] = {};
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return e;
  if (d < 0 || d >= 128) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[d]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    addr[d] = p;
  }
  *absmax = static_cast<float*>(addr[d]);
  *bins = static_cast<char*>(addr[d]) + kNoAllocBinsOffset;
  return cudaSuccess;
}

// ------------------------------------------------------------------ launchers
static int grid_for(int64_t work_items, int per_cta, int max_ctas) {
  int64_t g = (work_items + per_cta - 1) / per_cta;
  if (g < 1) g = 1;
  if (g > max_ctas) g = max_ctas;
  return static_cast<int>(g);
}

cudaError_t launch_nf4_quantize(const void* w, int w_dtype, int64_t n_elems, uint8_t* codes, float* absmax,
                                int8_t* absq, float* step, float* mean, void* ws_bins, unsigned* status,
                                int num_sms, cudaStream_t s) {
  const int64_t n_a = n_elems / 64;
  const int64_t n_groups = (n_a + 255) / 256;
  // bins (256 x u64) + counter; zeroed every call
  unsigned long long* bins = static_cast<unsigned long long*>(ws_bins);
  unsigned* counter = reinterpret_cast<unsigned*>(bins + 256);
  cudaError_t e = cudaMemsetAsync(ws_bins, 0, 256 * sizeof(unsigned long long) + 16, s);
  if (e != cudaSuccess) return e;
  const int g1 = grid_for((n_elems + 255) / 256, 8, num_sms * 8);
  if (w_dtype == 0)
    k_nf4_quantize<float><<<g1, 256, 0, s>>>(static_cast<const float*>(w), n_elems, codes, absmax, status);
  else
    k_nf4_quantize<__nv_bfloat16><<<g1, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w), n_elems, codes,
                                                      absmax, status);
  const int g2 = grid_for(n_a, 256 * 4, num_sms * 2);
  k_absmax_mean<<<g2, 256, 0, s>>>(absmax, n_a, bins, counter, mean, status);
  k_absmax_dq<<<static_cast<unsigned>(n_groups), 256, 0, s>>>(absmax, n_a, mean, absq, step);
  return cudaGetLastError();
}

cudaError_t launch_nf4_dequantize(const uint8_t* codes, const int8_t* absq, const float* step, const float* mean,
                                  uint16_t* out, int64_t n_elems, int num_sms, cudaStream_t s) {
  const int64_t n_blocks = n_elems / 64;
  const int g = grid_for((n_blocks + 31) / 32, 8, num_sms * 8);
  k_nf4_dequantize<<<g, 256, 0, s>>>(codes, absq, step, mean, out, n_blocks);
  return cudaGetLastError();
}

}  // namespace qlora
