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
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace qlora {

// ------------------------------------------------------------------ encode thresholds
// Threshold t_j (j = 0..14): the smallest float x with |x - L[j+1]| < |x - L[j]|
// in float32 arithmetic.  For x between the two levels both distances are
// monotone in x, so "x is strictly nearer to L[j+1]" switches exactly once and
// a bisection over the ordered floats finds the switch.  Then the nearest
// level with ties to the lower index is code(x) = #{ j : x >= t_j }.  Computed
// once on the host (each step is a single rounded float subtraction, the same
// on either side) and handed to the kernels.
static float host_bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static uint32_t host_f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}
// Monotone integer key of a float (total order of non-NaN floats, -0 == +0).
static int32_t host_f32_key(float f) {
  const int32_t b = static_cast<int32_t>(host_f32_bits(f));
  return b >= 0 ? b : -(b & 0x7fffffff);
}
static float host_key_f32(int32_t k) {
  return k >= 0 ? host_bits_f32(static_cast<uint32_t>(k)) : host_bits_f32(static_cast<uint32_t>(-k) | 0x80000000u);
}
static float host_nf4_threshold(int j) {
  static const uint32_t hex[16] = QLORA_NF4_LEVELS_HEX;
  const float lo = host_bits_f32(hex[j]), hi = host_bits_f32(hex[j + 1]);
  int32_t a = host_f32_key(lo), b = host_f32_key(hi);  // predicate false at a, true at b
  while (b - a > 1) {
    const int32_t mid = a + (b - a) / 2;
    const volatile float x = host_key_f32(mid);
    const volatile float d_hi = hi - x, d_lo = x - lo;
    if (d_hi < d_lo) b = mid; else a = mid;
  }
  return host_key_f32(b);
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

// ------------------------------------------------------------------ code lookup without a quotient
// The code of w in a block of absmax a is code(x), x = RN(w / a) in [-1, 1].
//
// Bucket.  g = round(16 x' + 16) in [0, 32] for an approximate x' = w * (1/a),
// taken from the bits of one FMA, 2^23 + 16 + w * (16/a).  Consecutive NF4
// thresholds t_j are at least 0.08 apart and a bucket is 1/16 wide, so a bucket
// holds at most one threshold; every threshold is more than 0.004 away from a
// bucket edge, far beyond the error of x', so the bucket of x' is a bucket that
// x itself may use:  code(x) = base[g] + [x >= t_b],  b = base[g] = #{j :
// bucket(t_j) < g}.
//
// Decision without dividing (bf16 weights).  RN(w / a) >= t exactly when
// w / a > m, m the midpoint between t and the float below it (w / a never
// equals m: that needs a 25-bit significand from 24-bit operands).  With
// h = (t - pred(t)) / 2 (a power of two), w - a m = (w - a t) + a h, and the
// FMA pair RN(RN(w - a t) + a h) has its sign.  For bf16 w and a (8-bit
// significands) a nonzero w - a m is a multiple of 2^(e_a + e_m - 31), at
// least a |m| 2^-33, while near the threshold w - a t is exact and the
// roundings stay below a |t| 2^-44.  (With 24-bit fp32 operands the grid is
// 2^-49 and the sign can flip, so fp32 weights take the IEEE quotient and only
// the bucket lookup.)  The low four bits of h's float hold the base code b
// (h's significand bits are zero; the perturbation is below 2^-19 relative).
// Valid while a h and w - a t stay normal and a t finite:
// 2^-90 <= a < 2^120; other blocks take the IEEE quotient and compare tree.
constexpr int kQzBuckets = 34;  // bucket 33 is a spare copy of 32
constexpr float kQzBucketBase = 8388624.f;  // 2^23 + 16
constexpr uint32_t kQzBucketBias = 0x4B000000u;  // bits of 2^23

__device__ __forceinline__ bool qz_fast_block(uint32_t a_bits) {
  return a_bits >= 0x12800000u && a_bits < 0x7b800000u;  // 2^-90 <= a < 2^120
}

// The 32-bit shared address of the entry is (bucket bits << 8) + the lane's
// base: the bits of 2^23 shifted by 8 leave nothing in the low 32 bits.
__device__ __forceinline__ uint32_t qz_code(float w, float a, float r16, uint32_t lane_tab) {
  const uint32_t addr = (__float_as_uint(__fmaf_rn(w, r16, kQzBucketBase)) << 8) + lane_tab;
  uint32_t t_bits, meta;
  asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(t_bits), "=r"(meta) : "r"(addr));
  const float d = __fmaf_rn(a, __uint_as_float(meta), __fmaf_rn(-a, __uint_as_float(t_bits), w));
  return (meta & 15u) + (d > 0.f ? 1u : 0u);
}

// The code of an exact x = RN(w / a), |x| <= 1, from the same table.
__device__ __forceinline__ uint32_t qz_code_x(float x, uint32_t lane_tab) {
  const uint32_t addr = (__float_as_uint(__fmaf_rn(x, 16.f, kQzBucketBase)) << 8) + lane_tab;
  uint32_t t_bits, meta;
  asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(t_bits), "=r"(meta) : "r"(addr));
  return (meta & 15u) + (x >= __uint_as_float(t_bits) ? 1u : 0u);
}

// Kernel parameter: the table {t_b bits, h_b bits | b} per bucket and the 15
// thresholds (for blocks outside the fast range).  Built once on the host.
struct QzParams {
  uint2 tab[kQzBuckets];
  float thr[16];
};

static QzParams host_build_qz_params() {
  QzParams p = {};
  for (int j = 0; j < 15; ++j) p.thr[j] = host_nf4_threshold(j);
  p.thr[15] = host_bits_f32(0x7f800000u);
  for (uint32_t g = 0; g < static_cast<uint32_t>(kQzBuckets); ++g) {
    uint32_t base = 0;
    for (int j = 0; j < 15; ++j)
      base += (host_f32_bits(std::fmaf(p.thr[j], 16.f, kQzBucketBase)) - kQzBucketBias) < g ? 1u : 0u;
    float t = host_bits_f32(0x7f800000u), h = 0x1p-30f;  // base 15: nothing above, the decision is always false
    if (base < 15) {
      t = p.thr[base];
      const uint32_t tb = host_f32_bits(t);
      const float below = host_bits_f32(t > 0.f ? tb - 1u : tb + 1u);  // thresholds are nonzero
      const volatile float diff = t - below;                            // exact (Sterbenz)
      h = diff * 0.5f;
    }
    p.tab[g] = make_uint2(host_f32_bits(t), host_f32_bits(h) | base);
  }
  return p;
}

static const QzParams& qz_params() {
  static const QzParams p = host_build_qz_params();
  return p;
}

// Replicates the table into shared memory, one copy per lane.
__device__ __forceinline__ void qz_fill_table(uint2* tab, const QzParams& qp) {
  for (int i = threadIdx.x; i < kQzBuckets * 32; i += blockDim.x) tab[i] = qp.tab[i >> 5];
}

// ------------------------------------------------------------------ exact-mean bins, register window
// Each block absmax a = m * 2^(max(e,1) - 150) (e the exponent field, m the
// significand with its hidden bit) adds m to bin e.  A lane keeps four
// consecutive bins in registers (the window opens at the first exponent it
// sees, minus one); other exponents go straight to the CTA's shared bins.
struct BinWindow {
  uint32_t lo = 0xffffffffu;
  unsigned long long b0 = 0, b1 = 0, b2 = 0, b3 = 0;
  __device__ __forceinline__ void add(uint32_t e, uint32_t m, unsigned long long* s_bins) {
    if (lo == 0xffffffffu) lo = e > 0 ? e - 1 : 0;
    const uint32_t d = e - lo;
    if (d < 4) {
      b0 += d == 0 ? m : 0u;
      b1 += d == 1 ? m : 0u;
      b2 += d == 2 ? m : 0u;
      b3 += d == 3 ? m : 0u;
    } else {
      atomicAdd(s_bins + e, static_cast<unsigned long long>(m));
    }
  }
  __device__ __forceinline__ void flush(unsigned long long* s_bins) const {
    if (lo == 0xffffffffu) return;
    const unsigned long long v[4] = {b0, b1, b2, b3};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (v[i] && lo + i < 255) atomicAdd(s_bins + lo + i, v[i]);
  }
};

// ------------------------------------------------------------------ exact mean of the absmax values
// The mean is float32( RN64(sum a_i) / n ) where RN64(sum) is the exactly
// rounded float64 value of the exact sum, so it does not depend on the order
// in which blocks are visited.  The exact sum is accumulated as integers: a
// float32 a = m * 2^(max(e,1) - 150) (m the 24-bit significand, e the biased
// exponent field), so sum_i a_i = sum_e B[e] * 2^(max(e,1) - 150) with
// B[e] = sum of m over values with exponent field e (64-bit, exact for up to
// 2^40 values).  One warp turns the bins into a 384-bit integer (sum * 2^149)
// and rounds it once to float64 (round to nearest, ties to even).
__device__ float exact_mean_from_bins(const unsigned long long* bins, int64_t n_a) {  // one full warp; global bins
  const int lane = threadIdx.x & 31;
  unsigned long long bv[8];  // bins 32 r + lane
  unsigned nz[8];            // their nonzero masks
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int e = r * 32 + lane;
    bv[r] = e < 255 ? __ldcg(bins + e) : 0ull;
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) nz[r] = __ballot_sync(0xffffffffu, bv[r] != 0);
  uint64_t limb[6] = {0, 0, 0, 0, 0, 0};  // little-endian; indexed statically only (stays in registers)
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    for (unsigned m = nz[r]; m; m &= m - 1) {
      const int src = __ffs(m) - 1;
      const int e = r * 32 + src;
      const uint64_t v = __shfl_sync(0xffffffffu, bv[r], src);
      const int sh = (e < 1 ? 1 : e) - 1;  // 0..253
      const int li = sh >> 6, bo = sh & 63;
      const uint64_t lo = v << bo, hi = bo ? (v >> (64 - bo)) : 0;  // hi < 2^63
      uint64_t carry = 0;
#pragma unroll
      for (int t = 0; t < 6; ++t) {
        const uint64_t add = (t == li ? lo : 0) + (t == li + 1 ? hi : 0);  // never both: no overflow
        const uint64_t s1 = limb[t] + add;
        const uint64_t c1 = s1 < add ? 1 : 0;
        const uint64_t s2 = s1 + carry;
        carry = c1 + (s2 < carry ? 1 : 0);
        limb[t] = s2;
      }
    }
  }
  int top = -1;  // most significant set bit
#pragma unroll
  for (int t = 0; t < 6; ++t)
    if (limb[t]) top = t * 64 + 63 - __clzll(static_cast<long long>(limb[t]));
  // 64 bits from bit `pos` up (pos >= 0)
  auto bits64 = [&](int pos) -> uint64_t {
    const int li = pos >> 6, bo = pos & 63;
    uint64_t r = 0;
#pragma unroll
    for (int t = 0; t < 6; ++t) {
      if (t == li) r |= limb[t] >> bo;
      if (t == li + 1 && bo) r |= limb[t] << (64 - bo);
    }
    return r;
  };
  double sum = 0.0;
  if (top >= 0 && top <= 52) {
    sum = ldexp(static_cast<double>(limb[0]), -149);  // < 2^53: exact
  } else if (top > 52) {
    const int shift = top - 52;  // keep bits [shift, top]
    uint64_t mant = bits64(shift) & ((1ull << 53) - 1);
    const bool round = (bits64(shift - 1) & 1ull) != 0;
    const int sp = shift - 1, sli = sp >> 6, sbo = sp & 63;  // sticky: any bit below shift - 1
    bool sticky = false;
#pragma unroll
    for (int t = 0; t < 6; ++t) {
      if (t < sli) sticky |= limb[t] != 0;
      if (t == sli && sbo) sticky |= (limb[t] & ((1ull << sbo) - 1)) != 0;
    }
    int exp2 = shift - 149;
    if (round && (sticky || (mant & 1ull))) {
      mant += 1;
      if (mant == (1ull << 53)) {
        mant >>= 1;
        exp2 += 1;
      }
    }
    sum = ldexp(static_cast<double>(mant), exp2);
  }
  return n_a > 0 ? __double2float_rn(__ddiv_rn(sum, static_cast<double>(n_a))) : 0.f;
}

// ------------------------------------------------------------------ quantise: shared pieces
// The block absmax values go into the exponent bins of the exact mean.
__device__ __forceinline__ void bin_block_absmax(uint32_t mb, BinWindow& win, unsigned long long* s_bins,
                                                 unsigned* status) {
  const uint32_t e = mb >> 23;
  if (e >= 255) {
    latch_status(status, ST_NONFINITE);
  } else {
    const uint32_t m = (e == 0) ? (mb & 0x7fffffu) : ((mb & 0x7fffffu) | 0x800000u);
    if (m) win.add(e, m, s_bins);
  }
}

// Adds the CTA's bins to the global bins; the last CTA to finish turns them
// into the mean (the double quantisation kernel that follows needs it).
__device__ void quant_bins_flush(const BinWindow& win, unsigned long long* s_bins, unsigned long long* bins,
                                 unsigned* counter, float* mean_out, int64_t n_a) {
  __shared__ int s_last;
  griddep_launch_dependents();  // the double quantisation waits for this whole grid anyway
  win.flush(s_bins);
  __syncthreads();
  for (int i = threadIdx.x; i < 256; i += blockDim.x)
    if (s_bins[i]) atomicAdd(bins + i, s_bins[i]);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(counter, 1u) == gridDim.x - 1);
  __syncthreads();
  if (s_last && threadIdx.x < 32) {
    __threadfence();
    const float m = exact_mean_from_bins(bins, n_a);
    if (threadIdx.x == 0) *mean_out = m;
  }
}

__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// max(|x|, |y|) of each bf16 half (the sign bit of the result is not the
// magnitude's and gets masked off); NaN propagates.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t x, uint32_t y) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
  return r;
}

// Codes of a bf16 block outside the fast range (zero, tiny or huge absmax,
// or not finite): IEEE quotient and the threshold compare tree.  Out of line:
// it is rare and its unrolled body would crowd the instruction cache.
struct Codes64 {
  uint4 lo, hi;  // packed codes of elements 0..31 and 32..63
};
__device__ __noinline__ Codes64 qz_slow_block(const uint8_t* row, int lane, float a, uint32_t mb,
                                              const QzParams& qp) {
  uint32_t packed[8];
  Thresholds th;
#pragma unroll
  for (int t = 0; t < 15; ++t) th.t[t] = qp.thr[t];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 q = *reinterpret_cast<const uint4*>(row + ((c ^ (lane & 7)) << 4));
    const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
    uint32_t pk = 0;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float x0 = (mb == 0) ? 0.f : __fdiv_rn(__uint_as_float(wv[h] << 16), a);
      const float x1 = (mb == 0) ? 0.f : __fdiv_rn(__uint_as_float(wv[h] & 0xffff0000u), a);
      pk |= nf4_code(th, x0) << (h * 8 + 4);
      pk |= nf4_code(th, x1) << (h * 8);
    }
    packed[c] = pk;
  }
  return {make_uint4(packed[0], packed[1], packed[2], packed[3]), make_uint4(packed[4], packed[5], packed[6], packed[7])};
}

// ------------------------------------------------------------------ quantise, bf16 weights
// One 64-block per lane.  The weight is viewed as rows of one block (128
// bytes); each warp streams boxes of 32 rows (4 KB) by TMA, 128-byte swizzled,
// through its own ring of kQbStages slots, lane 0 keeping kQbStages - 1 boxes
// in flight.  Lane L reads row L: its 16-byte chunk c sits at c ^ (L & 7), so
// the eight lanes of each quarter-warp hit eight different chunk positions.
constexpr int kQbWarps = 6;
constexpr int kQbThreads = kQbWarps * 32;
constexpr int kQbStages = 4;
constexpr int kQbBox = 32 * 128;
constexpr int kQbCtasPerSm = 2;
constexpr size_t kQbSmem = 1024 + static_cast<size_t>(kQbWarps) * kQbStages * kQbBox;  // + alignment slack

__global__ void __launch_bounds__(kQbThreads, kQbCtasPerSm)
    k_nf4_quantize_bf16(const __grid_constant__ CUtensorMap tm_w,  // [n_blocks rows x 64] bf16, box 64 x 32
                        int64_t n_blocks, uint8_t* __restrict__ codes, float* __restrict__ absmax,
                        unsigned long long* bins, unsigned* counter, float* mean_out, unsigned* status,
                        uint64_t wait_ns, const __grid_constant__ QzParams qp) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring_all = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(16) uint2 s_tab[kQzBuckets * 32];
  __shared__ unsigned long long s_bins[256];
  __shared__ uint64_t s_full[kQbWarps][kQbStages];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n_chunks = (n_blocks + 31) / 32;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kQbWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kQbWarps + warp;
  const int64_t my_chunks = first < n_chunks ? (n_chunks - first + warps_total - 1) / warps_total : 0;
  uint8_t* ring = ring_all + static_cast<size_t>(warp) * kQbStages * kQbBox;
  uint64_t* full = s_full[warp];
  auto issue = [&](int64_t j) {  // box j of this warp into slot j % kQbStages (rows past the end read as zero)
    uint64_t* bar = &full[j % kQbStages];
    mbar_arrive_expect_tx(bar, kQbBox);
    tma_load_2d(ring + (j % kQbStages) * kQbBox, &tm_w, bar, 0, static_cast<int>((first + j * warps_total) * 32));
  };
  if (lane == 0) {
    for (int st = 0; st < kQbStages; ++st) mbar_init(&full[st], 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tm_w);
    for (int64_t j = 0; j < kQbStages - 1 && j < my_chunks; ++j) issue(j);
  }
  for (int i = tid; i < 256; i += blockDim.x) s_bins[i] = 0;
  qz_fill_table(s_tab, qp);
  __syncthreads();
  const uint32_t lane_tab = smem_u32(s_tab) + static_cast<uint32_t>(lane) * 8u;

  BinWindow win;
  int64_t issued = my_chunks < kQbStages - 1 ? my_chunks : kQbStages - 1;
  int64_t j = 0;
  for (; j < my_chunks; ++j) {
    if (lane == 0 && issued < my_chunks) {  // refill the slot freed one trip ago
      fence_proxy_async_smem();
      issue(issued);
      ++issued;
    }
    const int st = static_cast<int>(j % kQbStages);
    if (!mbar_wait(&full[st], static_cast<uint32_t>((j / kQbStages) & 1), wait_ns, nullptr)) {
      latch_status(status, ST_TIMEOUT);
      break;
    }
    const uint8_t* row = ring + st * kQbBox + lane * 128;
    uint4 q[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) q[c] = *reinterpret_cast<const uint4*>(row + ((c ^ (lane & 7)) << 4));
    uint32_t m2[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) m2[c] = absmax_bf16x2(absmax_bf16x2(q[c].x, q[c].y), absmax_bf16x2(q[c].z, q[c].w));
#pragma unroll
    for (int c = 0; c < 4; ++c) m2[c] = absmax_bf16x2(m2[c], m2[c + 4]);
    const uint32_t m1 = absmax_bf16x2(absmax_bf16x2(m2[0], m2[1]), absmax_bf16x2(m2[2], m2[3]));
    const uint32_t mb = max(m1 & 0x7fffu, (m1 >> 16) & 0x7fffu) << 16;  // |.| as float bits
    const float a = __uint_as_float(mb);
    uint4 lo, hi;  // packed codes of weights 0..31 and 32..63
    if (qz_fast_block(mb)) {
      const float r16 = __fdividef(16.f, a);
      uint32_t packed[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t wv[4] = {q[c].x, q[c].y, q[c].z, q[c].w};
        uint32_t by[4];  // byte h = code(weight 2h) in the high nibble, code(weight 2h + 1) in the low
#pragma unroll
        for (int h = 0; h < 4; ++h)
          by[h] = qz_code(__uint_as_float(wv[h] << 16), a, r16, lane_tab) * 16u +
                  qz_code(__uint_as_float(wv[h] & 0xffff0000u), a, r16, lane_tab);
        // the four bytes into one word with three byte permutes
        packed[c] = prmt(prmt(by[0], by[1], 0x0040u), prmt(by[2], by[3], 0x0040u), 0x5410u);
      }
      lo = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      hi = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    } else {
      const Codes64 sc = qz_slow_block(row, lane, a, mb, qp);
      lo = sc.lo;
      hi = sc.hi;
    }
    __syncwarp();  // every lane has read the slot before lane 0 refills it next trip
    const int64_t blk = (first + j * warps_total) * 32 + lane;
    if (blk < n_blocks) {
      uint4* dst = reinterpret_cast<uint4*>(codes + blk * 32);
      dst[0] = lo;
      dst[1] = hi;
      absmax[blk] = a;
      bin_block_absmax(mb, win, s_bins, status);
    }
  }
  // after an expired wait: let the copies this warp still has in flight land before the CTA exits
  for (; j < issued; ++j)
    if (!mbar_wait(&full[j % kQbStages], static_cast<uint32_t>((j / kQbStages) & 1), wait_ns, nullptr)) break;
  quant_bins_flush(win, s_bins, bins, counter, mean_out, n_blocks);
}

// ------------------------------------------------------------------ quantise, fp32 weights
// Persistent warps walk 2 KB chunks (two sub-tiles of 256 weights) through a
// per-warp ring of 1-D bulk copies; each lane quantises 8 consecutive weights
// (8 lanes share one 64-block) with the IEEE quotient and the bucket table.
constexpr int kQfThreads = 256;
constexpr int kQfWarps = kQfThreads / 32;
constexpr int kQfChunk = 2048;
constexpr int kQfStages = 4;
constexpr size_t kQfRingBytes = static_cast<size_t>(kQfWarps) * kQfStages * kQfChunk;

__global__ void __launch_bounds__(kQfThreads, 3) k_nf4_quantize_f32(const float* __restrict__ w, int64_t n_elems,
                                                                   uint8_t* __restrict__ codes,
                                                                   float* __restrict__ absmax, unsigned long long* bins,
                                                                   unsigned* counter, float* mean_out, unsigned* status,
                                                                   uint64_t wait_ns, const __grid_constant__ QzParams qp) {
  extern __shared__ __align__(128) uint8_t s_ring[];  // [warp][stage][kQfChunk]
  __shared__ __align__(16) uint2 s_tab[kQzBuckets * 32];
  __shared__ unsigned long long s_bins[256];
  __shared__ uint64_t s_full[kQfWarps][kQfStages];
  constexpr int kChunkElems = kQfChunk / 4;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n_chunks = (n_elems + kChunkElems - 1) / kChunkElems;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kQfWarps;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kQfWarps + warp;
  uint8_t* ring = s_ring + static_cast<size_t>(warp) * kQfStages * kQfChunk;
  uint64_t* full = s_full[warp];
  const int64_t my_chunks = first < n_chunks ? (n_chunks - first + warps_total - 1) / warps_total : 0;
  auto issue = [&](int64_t j) {  // chunk j of this warp into slot j % kQfStages
    const int64_t e0 = (first + j * warps_total) * kChunkElems;
    const int64_t ne = (n_elems - e0 < kChunkElems) ? (n_elems - e0) : kChunkElems;  // multiple of 64
    const uint32_t bytes = static_cast<uint32_t>(ne * 4);
    uint64_t* bar = &full[j % kQfStages];
    mbar_arrive_expect_tx(bar, bytes);
    bulk_copy_g2s(ring + (j % kQfStages) * kQfChunk, w + e0, bytes, bar);
  };
  if (lane == 0) {
    for (int st = 0; st < kQfStages; ++st) mbar_init(&full[st], 1);
    fence_mbarrier_init();
    for (int64_t j = 0; j < kQfStages - 1 && j < my_chunks; ++j) issue(j);
  }
  for (int i = tid; i < 256; i += blockDim.x) s_bins[i] = 0;
  qz_fill_table(s_tab, qp);
  __syncthreads();
  const uint32_t lane_tab = smem_u32(s_tab) + static_cast<uint32_t>(lane) * 8u;

  BinWindow win;
  int64_t issued = my_chunks < kQfStages - 1 ? my_chunks : kQfStages - 1;
  int64_t j = 0;
  for (; j < my_chunks; ++j) {
    if (lane == 0 && issued < my_chunks) {
      fence_proxy_async_smem();
      issue(issued);
      ++issued;
    }
    const int st = static_cast<int>(j % kQfStages);
    if (!mbar_wait(&full[st], static_cast<uint32_t>((j / kQfStages) & 1), wait_ns, nullptr)) {
      latch_status(status, ST_TIMEOUT);
      break;
    }
    const uint8_t* chunk = ring + st * kQfChunk;
    const int64_t c0 = first + j * warps_total;
#pragma unroll
    for (int u = 0; u < kQfChunk / 1024; ++u) {
      const int64_t e0 = c0 * kChunkElems + u * 256 + lane * 8;
      const uint4* src = reinterpret_cast<const uint4*>(chunk + u * 1024 + lane * 32);
      const uint4 p0 = src[0], p1 = src[1];  // bytes past a short last chunk are stale; their lanes stop below
      const float v[8] = {__uint_as_float(p0.x), __uint_as_float(p0.y), __uint_as_float(p0.z), __uint_as_float(p0.w),
                          __uint_as_float(p1.x), __uint_as_float(p1.y), __uint_as_float(p1.z), __uint_as_float(p1.w)};
      uint32_t mb = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) mb = max(mb, __float_as_uint(v[i]) & 0x7fffffffu);
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
      mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
      if (e0 >= n_elems) continue;  // whole 64-blocks: e0 < n  =>  e0 + 8 <= n
      const float a = __uint_as_float(mb);
      uint32_t packed = 0;
      if (qz_fast_block(mb)) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          packed |= qz_code_x(__fdiv_rn(v[i], a), lane_tab) << ((i >> 1) * 8 + ((i & 1) ? 0 : 4));
      } else {
        Thresholds th;
#pragma unroll
        for (int t = 0; t < 15; ++t) th.t[t] = qp.thr[t];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float x = (mb == 0) ? 0.f : __fdiv_rn(v[i], a);
          packed |= nf4_code(th, x) << ((i >> 1) * 8 + ((i & 1) ? 0 : 4));
        }
      }
      reinterpret_cast<uint32_t*>(codes)[e0 >> 3] = packed;
      if ((lane & 7) == 0) {
        absmax[e0 >> 6] = a;
        bin_block_absmax(mb, win, s_bins, status);
      }
    }
    __syncwarp();  // every lane has read the slot before lane 0 refills it next trip
  }
  for (; j < issued; ++j)
    if (!mbar_wait(&full[j % kQfStages], static_cast<uint32_t>((j / kQfStages) & 1), wait_ns, nullptr)) break;
  quant_bins_flush(win, s_bins, bins, counter, mean_out, n_elems / 64);
}

// One warp per group of 256 absmax values: step = max|a - mu| / 127,
// q = clamp(rint((a - mu) / step), -127, 127), q = 0 when step == 0.
__global__ void __launch_bounds__(256) k_absmax_dq(const float* __restrict__ absmax, int64_t n_a,
                                                   const float* __restrict__ mean, int8_t* __restrict__ q,
                                                   float* __restrict__ step) {
  griddep_wait();  // absmax and the mean come from the kernel before
  const int lane = threadIdx.x & 31;
  const int64_t n_groups = (n_a + 255) / 256;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * 8;
  const float mu = __ldcg(mean);
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5); g < n_groups; g += warps_total) {
    const int64_t i0 = g * 256 + lane * 8;
    float d[8];
    if (i0 + 8 <= n_a) {
      const float4 u = __ldcg(reinterpret_cast<const float4*>(absmax + i0));
      const float4 w = __ldcg(reinterpret_cast<const float4*>(absmax + i0) + 1);
      const float a[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) d[i] = __fsub_rn(a[i], mu);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) d[i] = (i0 + i < n_a) ? __fsub_rn(__ldcg(absmax + i0 + i), mu) : 0.f;
    }
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(d[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float st = __fdiv_rn(m, 127.0f);
    if (lane == 0) step[g] = st;
    uint32_t packed[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int qi = 0;
      if (st != 0.f) {
        float r = rintf(__fdiv_rn(d[i], st));
        r = fminf(fmaxf(r, -127.f), 127.f);
        qi = static_cast<int>(r);
      }
      packed[i >> 2] |= (static_cast<uint32_t>(qi) & 0xffu) << ((i & 3) * 8);
    }
    if (i0 + 8 <= n_a) {
      *reinterpret_cast<uint2*>(q + i0) = make_uint2(packed[0], packed[1]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i0 + i < n_a) q[i0 + i] = static_cast<int8_t>((packed[i >> 2] >> ((i & 3) * 8)) & 0xffu);
    }
  }
  // The record is complete once this grid has exited.  A kernel launched after it with programmatic
  // dependent launch may start when the last CTA exits and read the record before its own
  // griddepcontrol.wait (the decode kernel stages weights that early), so every thread makes its
  // stores performed device-wide before it exits.
  __threadfence();
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
                                uint64_t wait_ns, int num_sms, cudaStream_t s) {
  const int64_t n_a = n_elems / 64;
  const int64_t n_groups = (n_a + 255) / 256;
  // bins (256 x u64) + CTA counter; zeroed every call
  unsigned long long* bins = static_cast<unsigned long long*>(ws_bins);
  unsigned* counter = reinterpret_cast<unsigned*>(bins + 256);
  cudaError_t e = cudaMemsetAsync(ws_bins, 0, 256 * sizeof(unsigned long long) + 16, s);
  if (e != cudaSuccess) return e;
  if (w_dtype == 0) {
    const int g1 = grid_for((n_elems + kQfChunk / 4 - 1) / (kQfChunk / 4), kQfWarps, num_sms * 3);
    e = set_smem_limit_once(k_nf4_quantize_f32, kQfRingBytes);
    if (e != cudaSuccess) return e;
    k_nf4_quantize_f32<<<g1, kQfThreads, kQfRingBytes, s>>>(static_cast<const float*>(w), n_elems, codes, absmax, bins,
                                                            counter, mean, status, wait_ns, qz_params());
  } else {
    CUtensorMap tm;
    if (n_a >= (int64_t(1) << 31) || !make_tensor_map_bf16_2d(&tm, w, 64, static_cast<uint64_t>(n_a), 128, 64, 32))
      return cudaErrorInvalidValue;
    const int g1 = grid_for((n_a + 31) / 32, kQbWarps, num_sms * kQbCtasPerSm);
    e = set_smem_limit_once(k_nf4_quantize_bf16, kQbSmem);
    if (e != cudaSuccess) return e;
    k_nf4_quantize_bf16<<<g1, kQbThreads, kQbSmem, s>>>(tm, n_a, codes, absmax, bins, counter, mean, status, wait_ns,
                                                         qz_params());
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int g2 = grid_for(n_groups, 8, num_sms * 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g2);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_absmax_dq, static_cast<const float*>(absmax), n_a, static_cast<const float*>(mean),
                         absq, step);
  if (e != cudaSuccess) return e;
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
