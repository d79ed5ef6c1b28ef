// C entry points of libqlora_nf4.so (declared and documented in include/qlora_nf4.h):
// argument checks, workspace carving, the latched device status word.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "qlora_nf4.h"

// Latched device status bits of this module (one word per device).
static __device__ unsigned g_qlora_status;

namespace {

thread_local char t_last_error[512] = "";
std::atomic<unsigned long long> g_wait_ns{2000000000ull};

struct DevInfo {
  bool ready = false;
  int supported = 0;
  int num_sms = 0;
  unsigned* status = nullptr;
  // the backward's LoRA gradient kernel runs on this stream, beside the dX
  // GEMM of the caller's stream (fork after U, join before the call returns)
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex side_mu;
  // qlora_copy_many's copy streams (forked from the caller's stream, joined back)
  static constexpr int kCopyStreams = 4;
  cudaStream_t copy[kCopyStreams] = {};
  cudaEvent_t copy_fork = nullptr, copy_join[kCopyStreams] = {};
  std::mutex copy_mu;
};
std::mutex g_mu;
DevInfo g_dev[128];

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int device(DevInfo** out) {
  int d = 0;
  cudaError_t e = cudaGetDevice(&d);
  if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (d < 0 || d >= 128) return fail(QLORA_ERR_UNSUPPORTED, "device index %d", d);
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& di = g_dev[d];
  if (!di.ready) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
    di.supported = (major == 10 && minor == 3);
    di.num_sms = sms;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_qlora_status);
    if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
    di.status = static_cast<unsigned*>(p);
    if (di.supported) {
      e = cudaStreamCreateWithFlags(&di.side, cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&di.fork, cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&di.join, cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&di.copy_fork, cudaEventDisableTiming);
      for (int i = 0; i < DevInfo::kCopyStreams && e == cudaSuccess; ++i) {
        e = cudaStreamCreateWithFlags(&di.copy[i], cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&di.copy_join[i], cudaEventDisableTiming);
      }
      if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "side stream: %s", cudaGetErrorString(e));
    }
    di.ready = true;
  }
  if (!di.supported) return fail(QLORA_ERR_UNSUPPORTED, "the kernels are built for sm_103a only");
  *out = &di;
  return QLORA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

int cuda_ret(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return QLORA_OK;
  if (e == cudaErrorInvalidValue && qlora::tensor_map_error()[0])
    return fail(QLORA_ERR_CUDA, "%s: %s", what, qlora::tensor_map_error());
  return fail(QLORA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int check_weight(const qlora_nf4_weight* w) {
  if (!w) return fail(QLORA_ERR_INVALID_ARGUMENT, "weight record is NULL");
  if (!w->codes || !w->absmax_q || !w->absmax_step || !w->absmax_mean)
    return fail(QLORA_ERR_INVALID_ARGUMENT, "weight record has a NULL pointer");
  if (!aligned16(w->codes) || !aligned16(w->absmax_q))
    return fail(QLORA_ERR_INVALID_ARGUMENT, "weight codes / absmax_q must be 16-byte aligned");
  if (w->n <= 0 || w->k <= 0) return fail(QLORA_ERR_INVALID_ARGUMENT, "weight shape [%lld, %lld]", (long long)w->n, (long long)w->k);
  if (w->k % 64) return fail(QLORA_ERR_UNSUPPORTED, "k = %lld is not a multiple of 64", (long long)w->k);
  if (w->n % 8) return fail(QLORA_ERR_UNSUPPORTED, "n = %lld is not a multiple of 8", (long long)w->n);
  if (w->n >= (1ll << 31) || w->k >= (1ll << 31)) return fail(QLORA_ERR_UNSUPPORTED, "weight dimension >= 2^31");
  return QLORA_OK;
}

int check_rank(int r) {
  if (r < 1 || r > 128) return fail(QLORA_ERR_UNSUPPORTED, "rank r = %d (need 1 <= r <= 128)", r);
  return QLORA_OK;
}

// Bytes of one internal bf16 LoRA operand (sT or sU): m rows of lora_ld(r) columns.
size_t lora_operand_bytes(int64_t m, int r) { return align256(static_cast<size_t>(m) * qlora::lora_ld(r) * 2); }

int check_ptr(const void* p, const char* name) {
  if (!p) return fail(QLORA_ERR_INVALID_ARGUMENT, "%s is NULL", name);
  if (!aligned16(p)) return fail(QLORA_ERR_INVALID_ARGUMENT, "%s is not 16-byte aligned", name);
  return QLORA_OK;
}

// A forward of 1..16 tokens without dropout runs as a one-problem grouped decode launch (the
// weight stream kernel); larger ones go through the tensor-core GEMMs.
bool use_decode(int64_t m, int64_t k) { return m >= 1 && m <= 16 && k <= 131072; }
qlora::GroupedProblem decode_shape(int64_t m, int64_t n, int64_t k, int r) {
  qlora::GroupedProblem g{};
  g.w.n = n;
  g.w.k = k;
  g.m = static_cast<int>(m);
  g.r = r;
  return g;
}

struct FwdWs {
  size_t st, ld, gemm, total;
};
FwdWs fwd_ws(int64_t m, int64_t n, int64_t k, int r, int sms) {
  FwdWs w;
  if (m <= 0) {
    w.st = w.ld = w.gemm = w.total = 0;
    return w;
  }
  w.st = lora_operand_bytes(m, r);
  w.ld = align256(qlora::lora_down_workspace_bytes(static_cast<int>(m), static_cast<int>(k), r, sms));
  w.gemm = align256(qlora::fwd_gemm_workspace_bytes(static_cast<int>(m), static_cast<int>(n), static_cast<int>(k), sms));
  w.total = w.st + w.ld + w.gemm;
  if (use_decode(m, k)) {  // the decode plan reuses the same workspace (the dropout forward does not take it)
    const qlora::GroupedProblem g = decode_shape(m, n, k, r);
    const size_t dec = align256(qlora::decode_workspace_bytes(&g, 1, sms));
    if (dec > w.total) w.total = dec;
  }
  return w;
}

// The forward's LoRA down-projection runs as the tiled TMA kernel beside the CTA-pair GEMM.
bool use_side(int64_t m, int r) { return qlora::use_pair_gemm(static_cast<int>(m)) && qlora::lora_side_supported(r); }
// The backward's U = dY B, by shape:
//  * r <= 16 and more than 256 tokens in at most a wave of 64-row blocks: k_lora_down_ks, k split
//    over a cluster (each CTA stages only its slice of B, 128 KB of dY in flight per CTA);
//  * wide r, long n or few tokens: the TMA kernel beside the GEMMs, on a k-major copy of B;
//  * otherwise k_lora_down (persistent over 16-row tiles, B staged once per CTA).
enum UPath { U_KS, U_SIDE, U_DOWN };
UPath u_path(int64_t m, int64_t n, int r, int sms) {
  int splits = 0, cps = 0;
  if (m > 256 && qlora::lora_down_ks_plan(static_cast<int>(m), static_cast<int>(n), r, sms, &splits, &cps)) return U_KS;
  if (qlora::lora_side_supported(r) && n % 64 == 0 && (r > 16 || n > 4096 || m <= 256)) return U_SIDE;
  return U_DOWN;
}

struct BwdWs {
  size_t su, st, ld, lg, gemm, total;
};
BwdWs bwd_ws(int64_t m, int64_t n, int64_t k, int r, int sms) {
  BwdWs w;
  if (m <= 0) {
    w.su = w.st = w.ld = w.lg = w.gemm = w.total = 0;
    return w;
  }
  w.su = lora_operand_bytes(m, r);
  w.st = w.su;
  w.ld = align256(qlora::lora_down_workspace_bytes(static_cast<int>(m), static_cast<int>(n), r, sms));
  if (u_path(m, n, r, sms) == U_SIDE) {
    // B^T [r, n], then the split-k partials and counters of U = dY B
    const size_t bt = align256(static_cast<size_t>(r) * n * 2) +
                      align256(qlora::lora_side_bwd_workspace_bytes(static_cast<int>(m), static_cast<int>(n), r, sms));
    if (bt > w.ld) w.ld = bt;
  }
  w.lg = align256(qlora::lora_grads_workspace_bytes(static_cast<int>(m), static_cast<int>(n), static_cast<int>(k), r, sms));
  w.gemm = align256(qlora::bwd_gemm_workspace_bytes(static_cast<int>(m), static_cast<int>(n), static_cast<int>(k), sms));
  w.total = w.su + w.st + w.ld + w.lg + w.gemm;
  return w;
}

// ---------------------------------------------------------------- tracing
// Every launcher call made by the entry points is counted (kernels launched),
// and, while profiling is on, bracketed by two CUDA events on its stream.
enum ProfName : int {
  P_QUANTIZE = 0, P_DEQUANTIZE, P_LORA_DOWN, P_FWD_GEMM, P_BWD_GEMM, P_LORA_GRADS, P_SILU_FWD, P_SILU_BWD,
  P_SELFTEST, P_FWD_GROUPED, P_LORA_SIDE_FWD, P_MERGE, P_LOWRANK, P_ADAMW, P_DROPOUT, P_LORA_SIDE_BWD, P_TRANSPOSE,
  P_COUNT
};
const char* const kProfNames[P_COUNT] = {"nf4_quantize(3 kernels)", "nf4_dequantize", "lora_down", "fwd_gemm",
                                         "bwd_dx_gemm", "lora_grads", "silu_mul_fwd", "silu_mul_bwd",
                                         "wait_selftest", "fwd_grouped", "lora_side_fwd", "nf4_merge",
                                         "lowrank_update", "adamw", "dropout", "lora_side_bwd", "lora_b_transpose"};
std::atomic<unsigned long long> g_launches{0};
std::atomic<bool> g_prof_on{false};
struct ProfRec {
  int name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_free;
double g_prof_ms[P_COUNT] = {0};
long long g_prof_calls[P_COUNT] = {0};

cudaEvent_t prof_event() {
  if (!g_prof_free.empty()) {
    cudaEvent_t e = g_prof_free.back();
    g_prof_free.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

struct Span {
  int name;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  Span(int n, cudaStream_t st, int kernels) : name(n), s(st) {
    g_launches.fetch_add(static_cast<unsigned long long>(kernels));
    if (!g_prof_on.load()) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    a = prof_event();
    if (a) cudaEventRecord(a, s);
  }
  ~Span() {
    if (!a) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    cudaEvent_t b = prof_event();
    if (!b) return;
    cudaEventRecord(b, s);
    g_prof_recs.push_back(ProfRec{name, a, b});
  }
};

qlora::Nf4Dev to_dev(const qlora_nf4_weight* w) {
  qlora::Nf4Dev d;
  d.codes = w->codes;
  d.absq = w->absmax_q;
  d.step = w->absmax_step;
  d.mean = w->absmax_mean;
  d.n = w->n;
  d.k = w->k;
  return d;
}

}  // namespace

extern "C" {

int qlora_nf4_quantize_workspace_bytes(int64_t n, int64_t k, size_t* bytes) {
  if (!bytes) return fail(QLORA_ERR_INVALID_ARGUMENT, "bytes is NULL");
  if (n <= 0 || k <= 0 || k % 64) return fail(QLORA_ERR_INVALID_ARGUMENT, "shape [%lld, %lld]", (long long)n, (long long)k);
  *bytes = align256(static_cast<size_t>(n) * k / 64 * 4) + 256 * 8 + 256;
  return QLORA_OK;
}

int qlora_nf4_quantize(const void* w, int w_dtype, int64_t n, int64_t k, const qlora_nf4_weight* out,
                       void* workspace, size_t workspace_bytes, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if ((rc = check_weight(out))) return rc;
  if (out->n != n || out->k != k) return fail(QLORA_ERR_INVALID_ARGUMENT, "record shape differs from the weight shape");
  if ((rc = check_ptr(w, "w"))) return rc;
  if (w_dtype != QLORA_DTYPE_F32 && w_dtype != QLORA_DTYPE_BF16) return fail(QLORA_ERR_INVALID_ARGUMENT, "w_dtype %d", w_dtype);
  size_t need = 0;
  qlora_nf4_quantize_workspace_bytes(n, k, &need);
  if ((rc = check_ptr(workspace, "workspace"))) return rc;
  if (workspace_bytes < need) return fail(QLORA_ERR_INVALID_ARGUMENT, "workspace %zu < %zu bytes", workspace_bytes, need);
  float* absmax = static_cast<float*>(workspace);
  void* bins = static_cast<char*>(workspace) + align256(static_cast<size_t>(n) * k / 64 * 4);
  Span sp(P_QUANTIZE, static_cast<cudaStream_t>(stream), 3);
  return cuda_ret(qlora::launch_nf4_quantize(w, w_dtype == QLORA_DTYPE_F32 ? 0 : 1, n * k, out->codes, absmax,
                                             out->absmax_q, out->absmax_step, out->absmax_mean, bins, di->status,
                                             g_wait_ns.load(), di->num_sms, static_cast<cudaStream_t>(stream)),
                  "quantize");
}

int qlora_nf4_quantize_noalloc(const void* w, int w_dtype, int64_t n, int64_t k, const qlora_nf4_weight* out,
                               void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if ((rc = check_weight(out))) return rc;
  if (out->n != n || out->k != k) return fail(QLORA_ERR_INVALID_ARGUMENT, "record shape differs from the weight shape");
  if ((rc = check_ptr(w, "w"))) return rc;
  if (w_dtype != QLORA_DTYPE_F32 && w_dtype != QLORA_DTYPE_BF16) return fail(QLORA_ERR_INVALID_ARGUMENT, "w_dtype %d", w_dtype);
  if (n * k > qlora::noalloc_max_weights())
    return fail(QLORA_ERR_UNSUPPORTED,
                "n*k = %lld weights exceeds the fixed scratch of the no-allocation quantiser (%lld weights); "
                "use qlora_nf4_quantize with a caller workspace",
                (long long)(n * k), (long long)qlora::noalloc_max_weights());
  float* absmax = nullptr;
  void* bins = nullptr;
  cudaError_t e = qlora::noalloc_scratch(&absmax, &bins);
  if (e != cudaSuccess) return cuda_ret(e, "no-allocation scratch address");
  Span sp(P_QUANTIZE, static_cast<cudaStream_t>(stream), 3);
  return cuda_ret(qlora::launch_nf4_quantize(w, w_dtype == QLORA_DTYPE_F32 ? 0 : 1, n * k, out->codes, absmax,
                                             out->absmax_q, out->absmax_step, out->absmax_mean, bins, di->status,
                                             g_wait_ns.load(), di->num_sms, static_cast<cudaStream_t>(stream)),
                  "quantize (no allocation)");
}

int qlora_nf4_dequantize(const qlora_nf4_weight* w, uint16_t* out, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if ((rc = check_weight(w))) return rc;
  if ((rc = check_ptr(out, "out"))) return rc;
  Span sp(P_DEQUANTIZE, static_cast<cudaStream_t>(stream), 1);
  return cuda_ret(qlora::launch_nf4_dequantize(w->codes, w->absmax_q, w->absmax_step, w->absmax_mean, out,
                                               w->n * w->k, di->num_sms, static_cast<cudaStream_t>(stream)),
                  "dequantize");
}

int qlora_nf4_merge(const qlora_nf4_weight* w, const uint16_t* lora_a, const uint16_t* lora_b, int r, float alpha,
                    uint16_t* out, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if ((rc = check_weight(w))) return rc;
  if ((rc = check_rank(r))) return rc;
  if ((rc = check_ptr(lora_a, "lora_a")) || (rc = check_ptr(lora_b, "lora_b")) || (rc = check_ptr(out, "out"))) return rc;
  Span sp(P_MERGE, static_cast<cudaStream_t>(stream), 1);
  return cuda_ret(qlora::launch_nf4_merge(to_dev(w), reinterpret_cast<const __nv_bfloat16*>(lora_a),
                                          reinterpret_cast<const __nv_bfloat16*>(lora_b), r,
                                          alpha / static_cast<float>(r), reinterpret_cast<__nv_bfloat16*>(out),
                                          static_cast<cudaStream_t>(stream)),
                  "merge");
}

int qlora_lowrank_update(const void* w, int w_dtype, int64_t n, int64_t k, const qlora_nf4_weight* sub,
                         const uint16_t* lora_a, const uint16_t* lora_b, int r, float coef, float* out, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if ((rc = check_ptr(w, "w")) || (rc = check_ptr(out, "out"))) return rc;
  if (w_dtype != QLORA_DTYPE_F32 && w_dtype != QLORA_DTYPE_BF16) return fail(QLORA_ERR_INVALID_ARGUMENT, "w_dtype %d", w_dtype);
  if (n <= 0 || k <= 0) return fail(QLORA_ERR_INVALID_ARGUMENT, "shape [%lld, %lld]", (long long)n, (long long)k);
  if (k % 64) return fail(QLORA_ERR_UNSUPPORTED, "k = %lld is not a multiple of 64", (long long)k);
  if (n >= (1ll << 31) || k >= (1ll << 31)) return fail(QLORA_ERR_UNSUPPORTED, "dimension >= 2^31");
  if (sub) {
    if ((rc = check_weight(sub))) return rc;
    if (sub->n != n || sub->k != k) return fail(QLORA_ERR_INVALID_ARGUMENT, "record shape differs from the weight shape");
  }
  if (r < 0 || r > 128) return fail(QLORA_ERR_UNSUPPORTED, "rank r = %d (need 0 <= r <= 128)", r);
  if (r > 0 && ((rc = check_ptr(lora_a, "lora_a")) || (rc = check_ptr(lora_b, "lora_b")))) return rc;
  qlora::Nf4Dev d;
  if (sub) d = to_dev(sub);
  Span sp(P_LOWRANK, static_cast<cudaStream_t>(stream), 1);
  return cuda_ret(qlora::launch_lowrank_update(w, w_dtype == QLORA_DTYPE_BF16 ? 1 : 0, sub ? &d : nullptr,
                                               reinterpret_cast<const __nv_bfloat16*>(lora_a),
                                               reinterpret_cast<const __nv_bfloat16*>(lora_b), r, coef, out, n, k,
                                               static_cast<cudaStream_t>(stream)),
                  "lowrank update");
}

// Managed (paged) memory of [p, p + bytes) is migrated to `device` ahead of the kernel; other memory is left alone.
static cudaError_t prefetch_if_managed(const void* p, size_t bytes, int device, cudaStream_t s) {
  if (!p || bytes == 0) return cudaSuccess;
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // an unregistered host pointer: nothing to prefetch
    return cudaSuccess;
  }
  if (a.type != cudaMemoryTypeManaged) return cudaSuccess;
  cudaMemLocation loc = {};
  loc.type = cudaMemLocationTypeDevice;
  loc.id = device;
  return cudaMemPrefetchAsync(p, bytes, loc, 0, s);
}

int qlora_adamw_step(const qlora_adamw_tensor* tensors, int count, float lr, float beta1, float beta2, float eps,
                     float weight_decay, int64_t step, int flags, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if (count < 0 || (count > 0 && !tensors)) return fail(QLORA_ERR_INVALID_ARGUMENT, "tensors");
  if (step < 1) return fail(QLORA_ERR_INVALID_ARGUMENT, "step = %lld (the first step is 1)", (long long)step);
  if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) || !(eps > 0.f))
    return fail(QLORA_ERR_INVALID_ARGUMENT, "beta1 / beta2 must be in [0, 1), eps > 0");
  if (flags & ~QLORA_ADAMW_PREFETCH) return fail(QLORA_ERR_INVALID_ARGUMENT, "flags 0x%x", flags);
  if (count == 0) return QLORA_OK;
  std::vector<qlora::AdamwTensor> ts(static_cast<size_t>(count));
  for (int i = 0; i < count; ++i) {
    const qlora_adamw_tensor& t = tensors[i];
    if (t.numel < 0) return fail(QLORA_ERR_INVALID_ARGUMENT, "tensor %d: numel %lld", i, (long long)t.numel);
    if (t.numel > 0 && (!t.master || !t.grad || !t.exp_avg || !t.exp_avg_sq))
      return fail(QLORA_ERR_INVALID_ARGUMENT, "tensor %d: NULL pointer", i);
    ts[static_cast<size_t>(i)] = qlora::AdamwTensor{t.master, reinterpret_cast<__nv_bfloat16*>(t.param), t.grad,
                                                    t.exp_avg, t.exp_avg_sq, t.numel};
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (flags & QLORA_ADAMW_PREFETCH) {
    int dev = 0;
    cudaGetDevice(&dev);
    for (const auto& t : ts) {
      const size_t b4 = static_cast<size_t>(t.numel) * 4;
      cudaError_t e = prefetch_if_managed(t.master, b4, dev, s);
      if (e == cudaSuccess) e = prefetch_if_managed(t.exp_avg, b4, dev, s);
      if (e == cudaSuccess) e = prefetch_if_managed(t.exp_avg_sq, b4, dev, s);
      if (e == cudaSuccess) e = prefetch_if_managed(t.grad, b4, dev, s);
      if (e != cudaSuccess) return cuda_ret(e, "prefetch of paged optimizer state");
    }
  }
  const qlora::AdamwHyper h = qlora::adamw_hyper(lr, beta1, beta2, eps, weight_decay, step);
  Span sp(P_ADAMW, s, (count + 239) / 240);
  return cuda_ret(qlora::launch_adamw(ts.data(), count, h, di->num_sms, s), "adamw");
}

int qlora_linear_fwd_workspace_bytes(int64_t m, int64_t n, int64_t k, int r, size_t* bytes) {
  if (!bytes) return fail(QLORA_ERR_INVALID_ARGUMENT, "bytes is NULL");
  if (m < 0 || n <= 0 || k <= 0 || m >= (1ll << 31)) return fail(QLORA_ERR_INVALID_ARGUMENT, "shape");
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  *bytes = fwd_ws(m, n, k, r, di->num_sms).total;
  return QLORA_OK;
}

// The forward of qlora_linear_fwd and qlora_linear_fwd_dropout.  With a mask, the LoRA branch
// reads x_drop = x * mask (written here first) and T carries the factor 1 / (1 - p).
static int linear_fwd_impl(const uint16_t* x, int64_t m, const qlora_nf4_weight* w, const uint16_t* lora_a,
                           const uint16_t* lora_b, int r, float alpha, const uint8_t* mask, float p_drop,
                           uint16_t* x_drop, uint16_t* y, float* t_save, void* workspace, size_t workspace_bytes,
                           void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if ((rc = check_weight(w))) return rc;
  if ((rc = check_rank(r))) return rc;
  if (m < 0 || m >= (1ll << 31)) return fail(QLORA_ERR_INVALID_ARGUMENT, "m = %lld", (long long)m);
  if (m == 0) return QLORA_OK;
  if ((rc = check_ptr(x, "x")) || (rc = check_ptr(lora_a, "lora_a")) || (rc = check_ptr(lora_b, "lora_b")) ||
      (rc = check_ptr(y, "y")) || (rc = check_ptr(t_save, "t_save")))
    return rc;
  if (mask && ((rc = check_ptr(x_drop, "x_drop")) || (rc = check_ptr(mask, "mask")))) return rc;
  const FwdWs ws = fwd_ws(m, w->n, w->k, r, di->num_sms);
  if ((rc = check_ptr(workspace, "workspace"))) return rc;
  if (workspace_bytes < ws.total) return fail(QLORA_ERR_INVALID_ARGUMENT, "workspace %zu < %zu bytes", workspace_bytes, ws.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* base = static_cast<char*>(workspace);
  __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(base);
  const float scale = alpha / static_cast<float>(r);
  const int M = static_cast<int>(m), N = static_cast<int>(w->n), K = static_cast<int>(w->k);
  cudaError_t e;
  if (!mask && use_decode(m, w->k)) {
    qlora::GroupedProblem g = decode_shape(m, w->n, w->k, r);
    g.x = reinterpret_cast<const __nv_bfloat16*>(x);
    g.w = to_dev(w);
    g.lora_a = reinterpret_cast<const __nv_bfloat16*>(lora_a);
    g.lora_b = reinterpret_cast<const __nv_bfloat16*>(lora_b);
    g.alpha = alpha;
    g.y = reinterpret_cast<__nv_bfloat16*>(y);
    g.t_save = t_save;
    Span sp(P_FWD_GROUPED, s, 1);
    // the decode's two per-problem counters sit at the start of its plan and must start at zero
    e = cudaMemsetAsync(workspace, 0, 256, s);
    if (e == cudaSuccess) e = qlora::launch_decode(&g, 1, workspace, di->status, g_wait_ns.load(), di->num_sms, s);
    return cuda_ret(e, "fwd decode");
  }
  // the LoRA branch input: x, or x * mask under dropout (T then scaled by 1 / (1 - p))
  const uint16_t* xl = x;
  float t_scale = 1.0f;
  if (mask) {
    Span sp(P_DROPOUT, s, 1);
    e = qlora::launch_dropout_apply(x, mask, x_drop, m * w->k, di->num_sms, s);
    if (e != cudaSuccess) return cuda_ret(e, "dropout apply");
    xl = x_drop;
    t_scale = static_cast<float>(1.0 / (1.0 - static_cast<double>(p_drop)));
  }
  {
    // T = X A^T on the SMs the GEMM's last wave leaves idle; the GEMM starts
    // beside it and waits for T only before its LoRA k block
    const int cap = qlora::idle_sms_beside(qlora::fwd_gemm_ctas(M, N, K, di->num_sms), di->num_sms);
    if (use_side(M, r)) {
      Span sp(P_LORA_SIDE_FWD, s, 1);
      e = qlora::launch_lora_side_fwd(reinterpret_cast<const __nv_bfloat16*>(xl),
                                      reinterpret_cast<const __nv_bfloat16*>(lora_a), M, K, r, scale, t_save, st, cap,
                                      di->status, g_wait_ns.load(), s, t_scale);
    } else {
      Span sp(P_LORA_DOWN, s, 1);
      e = qlora::launch_lora_down(reinterpret_cast<const __nv_bfloat16*>(xl),
                                  reinterpret_cast<const __nv_bfloat16*>(lora_a), 1, M, K, r, scale, t_save, st,
                                  base + ws.st, cap, s, nullptr, nullptr, 0, 1.0f, t_scale);
    }
  }
  if (e != cudaSuccess) return cuda_ret(e, "lora_down");
  {
    Span sp(P_FWD_GEMM, s, 1);
    e = qlora::launch_fwd_gemm(reinterpret_cast<const __nv_bfloat16*>(x), M, to_dev(w), st,
                             reinterpret_cast<const __nv_bfloat16*>(lora_b), r, reinterpret_cast<__nv_bfloat16*>(y),
                             base + ws.st + ws.ld, di->status, g_wait_ns.load(), di->num_sms, s);
  }
  return cuda_ret(e, "fwd_gemm");
}

int qlora_linear_fwd(const uint16_t* x, int64_t m, const qlora_nf4_weight* w, const uint16_t* lora_a,
                     const uint16_t* lora_b, int r, float alpha, uint16_t* y, float* t_save, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return linear_fwd_impl(x, m, w, lora_a, lora_b, r, alpha, nullptr, 0.f, nullptr, y, t_save, workspace,
                         workspace_bytes, stream);
}

static int check_dropout(const uint8_t* mask, float p) {
  if (!mask) return fail(QLORA_ERR_INVALID_ARGUMENT, "mask is NULL");
  if (!(p >= 0.f && p < 1.f)) return fail(QLORA_ERR_INVALID_ARGUMENT, "dropout probability %g not in [0, 1)", (double)p);
  return QLORA_OK;
}

int qlora_linear_fwd_dropout(const uint16_t* x, int64_t m, const qlora_nf4_weight* w, const uint16_t* lora_a,
                             const uint16_t* lora_b, int r, float alpha, const uint8_t* mask, float p,
                             uint16_t* x_drop, uint16_t* y, float* t_save, void* workspace, size_t workspace_bytes,
                             void* stream) {
  const int rc = check_dropout(mask, p);
  if (rc) return rc;
  return linear_fwd_impl(x, m, w, lora_a, lora_b, r, alpha, mask, p, x_drop, y, t_save, workspace, workspace_bytes,
                         stream);
}

int qlora_dropout_mask(uint64_t seed, uint64_t offset, int64_t m, int64_t k, float p, uint8_t* mask, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if (m < 0 || k <= 0 || k % 64) return fail(QLORA_ERR_INVALID_ARGUMENT, "shape [%lld, %lld] (k %% 64 == 0)", (long long)m, (long long)k);
  if (!(p >= 0.f && p < 1.f)) return fail(QLORA_ERR_INVALID_ARGUMENT, "dropout probability %g not in [0, 1)", (double)p);
  if (m == 0) return QLORA_OK;
  if ((rc = check_ptr(mask, "mask"))) return rc;
  Span sp(P_DROPOUT, static_cast<cudaStream_t>(stream), 1);
  return cuda_ret(qlora::launch_dropout_mask(seed, offset, m * k, p, mask, di->num_sms, static_cast<cudaStream_t>(stream)),
                  "dropout mask");
}

int qlora_linear_bwd_workspace_bytes(int64_t m, int64_t n, int64_t k, int r, size_t* bytes) {
  if (!bytes) return fail(QLORA_ERR_INVALID_ARGUMENT, "bytes is NULL");
  if (m < 0 || n <= 0 || k <= 0 || m >= (1ll << 31)) return fail(QLORA_ERR_INVALID_ARGUMENT, "shape");
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  *bytes = bwd_ws(m, n, k, r, di->num_sms).total;
  return QLORA_OK;
}

// The backward of qlora_linear_bwd and qlora_linear_bwd_dropout.  With a mask, x is the
// dropped branch input x_drop of the forward, dA carries 1 / (1 - p), and the LoRA term of dX is
// added after the GEMM, masked.
static int linear_bwd_impl(const uint16_t* dy, const uint16_t* x, int64_t m, const qlora_nf4_weight* w,
                           const uint16_t* lora_a, const uint16_t* lora_b, int r, float alpha, const uint8_t* mask,
                           float p_drop, const float* t_save, uint16_t* dx, float* da, float* db, int flags,
                           void* workspace, size_t workspace_bytes, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if ((rc = check_weight(w))) return rc;
  if ((rc = check_rank(r))) return rc;
  if (m < 0 || m >= (1ll << 31)) return fail(QLORA_ERR_INVALID_ARGUMENT, "m = %lld", (long long)m);
  if (flags & ~(QLORA_ACCUM_DX | QLORA_ACCUM_DA | QLORA_ACCUM_DB)) return fail(QLORA_ERR_INVALID_ARGUMENT, "flags 0x%x", flags);
  if ((rc = check_ptr(da, "da")) || (rc = check_ptr(db, "db"))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (m == 0) {
    // no tokens: the gradients are zero (or unchanged when accumulating)
    cudaError_t e = cudaSuccess;
    if (!(flags & QLORA_ACCUM_DA)) e = cudaMemsetAsync(da, 0, static_cast<size_t>(r) * w->k * 4, s);
    if (e == cudaSuccess && !(flags & QLORA_ACCUM_DB)) e = cudaMemsetAsync(db, 0, static_cast<size_t>(w->n) * r * 4, s);
    return cuda_ret(e, "bwd m == 0");
  }
  if ((rc = check_ptr(dy, "dy")) || (rc = check_ptr(x, "x")) || (rc = check_ptr(lora_a, "lora_a")) ||
      (rc = check_ptr(lora_b, "lora_b")) || (rc = check_ptr(t_save, "t_save")) || (rc = check_ptr(dx, "dx")))
    return rc;
  const BwdWs ws = bwd_ws(m, w->n, w->k, r, di->num_sms);
  if ((rc = check_ptr(workspace, "workspace"))) return rc;
  if (workspace_bytes < ws.total) return fail(QLORA_ERR_INVALID_ARGUMENT, "workspace %zu < %zu bytes", workspace_bytes, ws.total);
  char* base = static_cast<char*>(workspace);
  __nv_bfloat16* su = reinterpret_cast<__nv_bfloat16*>(base);
  __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(base + ws.su);
  void* ldws = base + ws.su + ws.st;
  void* lgws = base + ws.su + ws.st + ws.ld;
  void* gemmws = base + ws.su + ws.st + ws.ld + ws.lg;
  const float scale = alpha / static_cast<float>(r);
  const float inv_keep = mask ? static_cast<float>(1.0 / (1.0 - static_cast<double>(p_drop))) : 1.0f;
  const int M = static_cast<int>(m), N = static_cast<int>(w->n), K = static_cast<int>(w->k);
  const uint64_t wait = g_wait_ns.load();
  const __nv_bfloat16* dyb = reinterpret_cast<const __nv_bfloat16*>(dy);
  const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(x);
  cudaError_t e;
  // U (all SMs) on the caller's stream, then the dX GEMM there (started early by
  // programmatic dependent launch, it waits for U only before its LoRA k block)
  // and, forked onto the side stream after U, the dA / dB kernel on the SMs the
  // GEMM leaves idle; the caller's stream waits for the side stream before the
  // call returns.
  const UPath up = u_path(M, N, r, di->num_sms);
  if (up == U_SIDE) {
    // B^T (a k-major copy of B) and, in the same launch, sT = bf16(s * t_save) and U's split
    // counters cleared; then U = dY B by the TMA kernel with k split over the SMs (the dX GEMM
    // launches as U's CTAs finish and waits for sU only before its LoRA k block)
    __nv_bfloat16* bt = static_cast<__nv_bfloat16*>(ldws);
    void* uws = static_cast<char*>(ldws) + align256(static_cast<size_t>(r) * N * 2);
    unsigned* cnt = qlora::lora_side_bwd_counters(uws, M, N, r, di->num_sms);
    {
      Span sp(P_TRANSPOSE, s, 1);
      e = qlora::launch_transpose_kr(reinterpret_cast<const __nv_bfloat16*>(lora_b), bt, N, r, di->num_sms, s, t_save,
                                     st, static_cast<int64_t>(M), scale, cnt, cnt ? (M + 127) / 128 : 0);
    }
    if (e == cudaSuccess) {
      Span sp(P_LORA_SIDE_BWD, s, 1);
      e = qlora::launch_lora_side_bwd(dyb, bt, M, N, r, scale, su, uws, di->num_sms, di->status, wait, s);
    }
  } else if (up == U_KS) {
    // U = dY B (B read as stored), k split over clusters, and in the same launch sT = bf16(s * t_save)
    Span sp(P_LORA_DOWN, s, 1);
    e = qlora::launch_lora_down_ks(dyb, reinterpret_cast<const __nv_bfloat16*>(lora_b), 0, M, N, r, scale, nullptr,
                                   su, di->num_sms, s, t_save, st, static_cast<int64_t>(M), scale);
  } else {
    // U = dY B (B read as stored) on all SMs and, in the same launch, sT = bf16(s * t_save)
    Span sp(P_LORA_DOWN, s, 1);
    e = qlora::launch_lora_down(dyb, reinterpret_cast<const __nv_bfloat16*>(lora_b), 0, M, N, r, scale, nullptr, su,
                                ldws, di->num_sms, s, t_save, st, static_cast<int64_t>(M), scale);
  }
  if (e != cudaSuccess) return cuda_ret(e, "lora_down (U)");
  std::lock_guard<std::mutex> lk(di->side_mu);
  e = cudaEventRecord(di->fork, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(di->side, di->fork, 0);
  if (e != cudaSuccess) return cuda_ret(e, "fork to the side stream");
  {
    Span sp(P_LORA_GRADS, di->side, 1);
    const int cap = qlora::idle_sms_beside(qlora::bwd_gemm_ctas(M, N, K, di->num_sms), di->num_sms);
    e = qlora::launch_lora_grads(xb, dyb, su, st, M, N, K, r, da, db, (flags & QLORA_ACCUM_DA) ? 1 : 0,
                                 (flags & QLORA_ACCUM_DB) ? 1 : 0, lgws, di->status, wait, cap, di->side, inv_keep);
  }
  cudaError_t ej = cudaEventRecord(di->join, di->side);
  if (e == cudaSuccess) {
    Span sp(P_BWD_GEMM, s, 1);
    e = qlora::launch_bwd_dx_gemm(dyb, M, to_dev(w), su, reinterpret_cast<const __nv_bfloat16*>(lora_a), r,
                                  reinterpret_cast<__nv_bfloat16*>(dx), (flags & QLORA_ACCUM_DX) ? 1 : 0, gemmws,
                                  di->status, wait, di->num_sms, s, mask ? 0 : 1);
  }
  if (e == cudaSuccess && mask) {
    Span sp(P_DROPOUT, s, 1);
    e = qlora::launch_dropout_lora_dx(reinterpret_cast<__nv_bfloat16*>(dx), su,
                                      reinterpret_cast<const __nv_bfloat16*>(lora_a), mask, M, K, r, inv_keep, s);
  }
  // always join, so a stream capture never ends with the side stream forked
  const cudaError_t ew = ej == cudaSuccess ? cudaStreamWaitEvent(s, di->join, 0) : ej;
  if (e == cudaSuccess) e = ew;
  return cuda_ret(e, "bwd dx gemm");
}

int qlora_linear_bwd(const uint16_t* dy, const uint16_t* x, int64_t m, const qlora_nf4_weight* w,
                     const uint16_t* lora_a, const uint16_t* lora_b, int r, float alpha, const float* t_save,
                     uint16_t* dx, float* da, float* db, int flags, void* workspace, size_t workspace_bytes,
                     void* stream) {
  return linear_bwd_impl(dy, x, m, w, lora_a, lora_b, r, alpha, nullptr, 0.f, t_save, dx, da, db, flags, workspace,
                         workspace_bytes, stream);
}

int qlora_linear_bwd_dropout(const uint16_t* dy, const uint16_t* x_drop, int64_t m, const qlora_nf4_weight* w,
                             const uint16_t* lora_a, const uint16_t* lora_b, int r, float alpha, const uint8_t* mask,
                             float p, const float* t_save, uint16_t* dx, float* da, float* db, int flags,
                             void* workspace, size_t workspace_bytes, void* stream) {
  const int rc = check_dropout(mask, p);
  if (rc) return rc;
  if (m > 0 && !aligned16(mask)) return fail(QLORA_ERR_INVALID_ARGUMENT, "mask is not 16-byte aligned");
  return linear_bwd_impl(dy, x_drop, m, w, lora_a, lora_b, r, alpha, mask, p, t_save, dx, da, db, flags, workspace,
                         workspace_bytes, stream);
}

// The grouped problems as the launcher sees them (shapes only are needed for the workspace plan).
static int grouped_problems(const qlora_linear_problem* problems, int count, std::vector<qlora::GroupedProblem>& gp,
                            bool check_pointers) {
  gp.assign(static_cast<size_t>(count), qlora::GroupedProblem{});
  int rc = 0;
  for (int i = 0; i < count; ++i) {
    const qlora_linear_problem& q = problems[i];
    if ((rc = check_weight(q.w))) return fail(rc, "problem %d: %s", i, t_last_error);
    if (q.m < 1 || q.m > 16) return fail(QLORA_ERR_UNSUPPORTED, "problem %d: m = %lld (the grouped path takes 1..16 tokens)", i, (long long)q.m);
    if (q.r < 1 || q.r > 128) return fail(QLORA_ERR_UNSUPPORTED, "problem %d: r = %d (need 1 <= r <= 128)", i, q.r);
    if (q.w->k > 131072)
      return fail(QLORA_ERR_UNSUPPORTED, "problem %d: k = %lld (the grouped path takes k <= 131072)", i,
                  (long long)q.w->k);
    if (check_pointers) {
      if ((rc = check_ptr(q.x, "x")) || (rc = check_ptr(q.lora_a, "lora_a")) || (rc = check_ptr(q.lora_b, "lora_b")) ||
          (rc = check_ptr(q.y, "y")))
        return fail(rc, "problem %d: %s", i, t_last_error);
      if (q.t_save && !aligned16(q.t_save)) return fail(QLORA_ERR_INVALID_ARGUMENT, "problem %d: t_save not 16-byte aligned", i);
    }
    qlora::GroupedProblem& g = gp[static_cast<size_t>(i)];
    g.x = reinterpret_cast<const __nv_bfloat16*>(q.x);
    g.w = to_dev(q.w);
    g.lora_a = reinterpret_cast<const __nv_bfloat16*>(q.lora_a);
    g.lora_b = reinterpret_cast<const __nv_bfloat16*>(q.lora_b);
    g.m = static_cast<int>(q.m);
    g.r = q.r;
    g.alpha = q.alpha;
    g.y = reinterpret_cast<__nv_bfloat16*>(q.y);
    g.t_save = q.t_save;
  }
  return QLORA_OK;
}

// Workspace of the launches: problems go out in chunks of at most
// decode_max_problems(), each chunk with its own plan.
static size_t grouped_workspace(const std::vector<qlora::GroupedProblem>& gp, int num_sms) {
  const int count = static_cast<int>(gp.size()), chunk = qlora::decode_max_problems();
  size_t tot = 0;
  for (int i0 = 0; i0 < count; i0 += chunk)
    tot += qlora::decode_workspace_bytes(gp.data() + i0, count - i0 < chunk ? count - i0 : chunk, num_sms);
  return tot;
}


int qlora_linear_fwd_grouped_workspace_bytes(const qlora_linear_problem* problems, int count, size_t* bytes) {
  if (!bytes) return fail(QLORA_ERR_INVALID_ARGUMENT, "bytes is NULL");
  if (count < 0 || (count > 0 && !problems)) return fail(QLORA_ERR_INVALID_ARGUMENT, "problems");
  *bytes = 0;
  if (count == 0) return QLORA_OK;
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  std::vector<qlora::GroupedProblem> gp;
  if ((rc = grouped_problems(problems, count, gp, false))) return rc;
  *bytes = grouped_workspace(gp, di->num_sms);
  return QLORA_OK;
}

int qlora_linear_fwd_grouped(const qlora_linear_problem* problems, int count, void* workspace, size_t workspace_bytes,
                             void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if (count < 0 || (count > 0 && !problems)) return fail(QLORA_ERR_INVALID_ARGUMENT, "problems");
  if (count == 0) return QLORA_OK;
  std::vector<qlora::GroupedProblem> gp;
  if ((rc = grouped_problems(problems, count, gp, true))) return rc;
  const size_t need = grouped_workspace(gp, di->num_sms);
  if ((rc = check_ptr(workspace, "workspace"))) return rc;
  if (workspace_bytes < need) return fail(QLORA_ERR_INVALID_ARGUMENT, "workspace %zu < %zu bytes", workspace_bytes, need);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int chunk = qlora::decode_max_problems();
  char* ws = static_cast<char*>(workspace);
  for (int i0 = 0; i0 < count; i0 += chunk) {
    const int n = count - i0 < chunk ? count - i0 : chunk;
    Span sp(P_FWD_GROUPED, s, 1);
    cudaError_t e = qlora::launch_decode(gp.data() + i0, n, ws, di->status, g_wait_ns.load(), di->num_sms, s);
    if (e != cudaSuccess) return cuda_ret(e, "fwd grouped");
    ws += qlora::decode_workspace_bytes(gp.data() + i0, n, di->num_sms);
  }
  return QLORA_OK;
}

int qlora_silu_mul_fwd(const uint16_t* g, const uint16_t* u, uint16_t* h, int64_t count, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if (count < 0 || (count & 1)) return fail(QLORA_ERR_INVALID_ARGUMENT, "count %lld must be even and >= 0", (long long)count);
  if (count == 0) return QLORA_OK;
  if ((rc = check_ptr(g, "g")) || (rc = check_ptr(u, "u")) || (rc = check_ptr(h, "h"))) return rc;
  Span sp(P_SILU_FWD, static_cast<cudaStream_t>(stream), 1);
  return cuda_ret(qlora::launch_silu_mul_fwd(g, u, h, count, di->num_sms, static_cast<cudaStream_t>(stream)), "silu fwd");
}

int qlora_silu_mul_bwd(const uint16_t* dh, const uint16_t* g, const uint16_t* u, uint16_t* dg, uint16_t* du,
                       int64_t count, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if (count < 0 || (count & 1)) return fail(QLORA_ERR_INVALID_ARGUMENT, "count %lld must be even and >= 0", (long long)count);
  if (count == 0) return QLORA_OK;
  if ((rc = check_ptr(dh, "dh")) || (rc = check_ptr(g, "g")) || (rc = check_ptr(u, "u")) || (rc = check_ptr(dg, "dg")) ||
      (rc = check_ptr(du, "du")))
    return rc;
  Span sp(P_SILU_BWD, static_cast<cudaStream_t>(stream), 1);
  return cuda_ret(qlora::launch_silu_mul_bwd(dh, g, u, dg, du, count, di->num_sms, static_cast<cudaStream_t>(stream)),
                  "silu bwd");
}

int qlora_get_status(void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  unsigned st = 0;
  e = cudaMemcpy(&st, di->status, sizeof(st), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (st) {
    const unsigned zero = 0;
    e = cudaMemcpy(di->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
  }
  if (st & qlora::ST_TIMEOUT) return fail(QLORA_ERR_TIMEOUT, "a bounded wait expired on the device");
  if (st & qlora::ST_NONFINITE) return fail(QLORA_ERR_NONFINITE, "non-finite weight seen by the quantiser");
  if (st) return fail(QLORA_ERR_CUDA, "device status 0x%x", st);
  return QLORA_OK;
}

const char* qlora_strerror(int code) {
  switch (code) {
    case QLORA_OK: return "ok";
    case QLORA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case QLORA_ERR_UNSUPPORTED: return "unsupported device or shape";
    case QLORA_ERR_CUDA: return "CUDA error";
    case QLORA_ERR_TIMEOUT: return "bounded device wait expired";
    case QLORA_ERR_NONFINITE: return "non-finite weight";
    default: return "unknown error code";
  }
}

const char* qlora_last_error(void) { return t_last_error; }

int qlora_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) return fail(QLORA_ERR_INVALID_ARGUMENT, "wait limit must be > 0");
  g_wait_ns.store(ns);
  return QLORA_OK;
}

int qlora_selftest_wait_timeout(uint64_t wait_ns, void* stream) {
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  if (wait_ns == 0 || wait_ns > 10000000000ull) return fail(QLORA_ERR_INVALID_ARGUMENT, "wait_ns out of range");
  Span sp(P_SELFTEST, static_cast<cudaStream_t>(stream), 1);
  return cuda_ret(qlora::launch_wait_selftest(di->status, wait_ns, static_cast<cudaStream_t>(stream)), "selftest");
}

unsigned long long qlora_launch_count(void) { return g_launches.load(); }

int qlora_profile_enable(int on) {
  g_prof_on.store(on != 0);
  return QLORA_OK;
}

int qlora_profile_collect(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (const ProfRec& r : g_prof_recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) == cudaSuccess && cudaEventElapsedTime(&ms, r.a, r.b) == cudaSuccess) {
      g_prof_ms[r.name] += ms;
      g_prof_calls[r.name] += 1;
    }
    g_prof_free.push_back(r.a);
    g_prof_free.push_back(r.b);
  }
  g_prof_recs.clear();
  return P_COUNT;
}

const char* qlora_profile_name(int i) { return (i >= 0 && i < P_COUNT) ? kProfNames[i] : ""; }

double qlora_profile_total_ms(int i) { return (i >= 0 && i < P_COUNT) ? g_prof_ms[i] : 0.0; }

long long qlora_profile_calls(int i) { return (i >= 0 && i < P_COUNT) ? g_prof_calls[i] : 0; }

int qlora_profile_reset(void) {
  qlora_profile_collect();
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (int i = 0; i < P_COUNT; ++i) {
    g_prof_ms[i] = 0.0;
    g_prof_calls[i] = 0;
  }
  return QLORA_OK;
}

int qlora_copy_many(const qlora_copy* copies, int count, void* stream) {
  if (count < 0 || (count > 0 && copies == nullptr)) return fail(QLORA_ERR_INVALID_ARGUMENT, "copy list");
  for (int i = 0; i < count; ++i)
    if (copies[i].bytes > 0 && (copies[i].dst == nullptr || copies[i].src == nullptr))
      return fail(QLORA_ERR_INVALID_ARGUMENT, "copy %d: NULL pointer", i);
  if (count == 0) return QLORA_OK;
  DevInfo* di = nullptr;
  int rc = device(&di);
  if (rc) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  constexpr size_t kMinPiece = size_t(2) << 20;
  constexpr int kN = DevInfo::kCopyStreams;
  std::lock_guard<std::mutex> lk(di->copy_mu);
  cudaError_t e = cudaEventRecord(di->copy_fork, s);
  for (int i = 0; i < kN && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(di->copy[i], di->copy_fork, 0);
  if (e != cudaSuccess) return cuda_ret(e, "fork to the copy streams");
  int next = 0;
  cudaError_t ec = cudaSuccess;
  for (int i = 0; i < count && ec == cudaSuccess; ++i) {
    const size_t bytes = copies[i].bytes;
    if (bytes == 0) continue;
    size_t pieces = bytes / kMinPiece;
    if (pieces < 1) pieces = 1;
    if (pieces > static_cast<size_t>(kN)) pieces = kN;
    const size_t per = ((bytes + pieces - 1) / pieces + 15) & ~size_t(15);
    for (size_t off = 0; off < bytes && ec == cudaSuccess; off += per) {
      const size_t len = bytes - off < per ? bytes - off : per;
      ec = cudaMemcpyAsync(static_cast<char*>(copies[i].dst) + off, static_cast<const char*>(copies[i].src) + off, len,
                           cudaMemcpyDefault, di->copy[next]);
      next = (next + 1) % kN;
    }
  }
  // always join, so a stream capture never ends with the copy streams forked
  cudaError_t ej = cudaSuccess;
  for (int i = 0; i < kN; ++i) {
    cudaError_t e1 = cudaEventRecord(di->copy_join[i], di->copy[i]);
    if (e1 == cudaSuccess) e1 = cudaStreamWaitEvent(s, di->copy_join[i], 0);
    if (ej == cudaSuccess) ej = e1;
  }
  if (ec != cudaSuccess) return cuda_ret(ec, "copy");
  return cuda_ret(ej, "join the copy streams");
}

int qlora_device_sm_count(void) {
  DevInfo* di = nullptr;
  if (device(&di)) return 0;
  return di->num_sms;
}

}  // extern "C"
