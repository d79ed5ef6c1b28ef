/*
 * qlora_nf4.h -- C ABI of libqlora_nf4.so: the QLoRA NF4 linear layer on one
 * B300 GPU (sm_103a).
 *
 * What it computes (sources cited by page title and section):
 *   - Ultralytics glossary "QLoRA", section "How QLoRA works": each weight is a
 *     4-bit code indexing one of 16 NF4 levels (normal quantiles with an exact
 *     zero, normalised to [-1, 1]); 64 weights share one absmax scale; the
 *     scales are quantised again to 8 bits in groups of 256 ("double
 *     quantisation"); the frozen layer dequantises to bfloat16 before the
 *     matmul, adds the LoRA output, and backpropagation updates only the two
 *     LoRA matrices.
 *   - Day 25 notes "Fine-tuning and LoRA/QLoRA", section 2.1: W = W0 + B A with
 *     B in R^{d x r}, A in R^{r x k}; section 6.2: scale s = alpha / r.
 *   - fedte.cc "QLoRA fine-tuning on 4 GB", section 1: 0.5 byte per parameter
 *     for the codes, one fp32 scale per 64 parameters before double quantisation.
 *
 * Conventions for every entry point:
 *   - All tensors are DEVICE pointers on the current CUDA device, row-major,
 *     16-byte aligned, allocated and owned by the caller.  The library never
 *     allocates or frees device memory.  Workspace sizes are queried with the
 *     *_workspace_bytes calls; workspaces need 256-byte alignment and may be
 *     reused between calls that are ordered on the same stream.
 *   - bfloat16 tensors are passed as uint16_t* (raw bf16 bits).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls are asynchronous on that stream and never synchronise the host,
 *     except qlora_get_status.  Calls on different streams may run at the same
 *     time when they use distinct workspaces and outputs (e.g. the gate and up
 *     forwards of an MLP block); the backward calls of a device share one
 *     internal stream for their dA / dB kernel, so those kernels of concurrent
 *     backward calls run one after the other.
 *   - The kernels are launched with programmatic dependent launch: a kernel may
 *     start before the one ahead of it on the stream has finished, and waits for
 *     it (griddepcontrol.wait) before touching its outputs.  Every kernel of the
 *     library lets the next one start only after that wait, and the first kernel
 *     of a forward call reads only the NF4 record before it.  So a caller's own
 *     kernel that writes the record (or anything a call reads) must not let the
 *     next kernel of the stream launch early (griddepcontrol.launch_dependents)
 *     before those writes are done; ordinary launches never do.
 *   - Argument errors are returned synchronously, before anything is launched.
 *     Errors found on the device (a bounded wait that expired, a non-finite
 *     weight) are latched in a per-device status word and returned by
 *     qlora_get_status.
 *   - Shapes: W is [n, k] (out x in, as a PyTorch Linear); k % 64 == 0
 *     (a block of 64 never crosses a row); tokens m >= 0 (m == 0 is a no-op);
 *     LoRA rank 1 <= r <= 128 (Day 25 notes, section 6.2: r is a free
 *     hyper-parameter, 4 to 64 typical); all of m, n, k < 2^31.
 *     n % 8 == 0 as well: the activations Y and dY have n columns and are read
 *     and written by the Tensor Memory Accelerator, whose row pitch must be a
 *     multiple of 16 bytes (n bf16 values).  Every Llama projection satisfies
 *     both (n, k in {4096, 8192, 11008, 22016}).
 */
#ifndef QLORA_NF4_H_
#define QLORA_NF4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ----------------------------------------------------------------- return codes */
#define QLORA_OK 0
#define QLORA_ERR_INVALID_ARGUMENT 1 /* null / misaligned pointer, bad shape or dtype */
#define QLORA_ERR_UNSUPPORTED 2      /* not an sm_103 device, or a shape outside the limits above */
#define QLORA_ERR_CUDA 3             /* a CUDA launch or runtime call failed (see qlora_last_error) */
#define QLORA_ERR_TIMEOUT 4          /* a kernel's bounded wait expired (device status) */
#define QLORA_ERR_NONFINITE 5        /* NaN / Inf weight seen by the quantiser (device status) */

/* ----------------------------------------------------------------- dtypes and flags */
#define QLORA_DTYPE_F32 0
#define QLORA_DTYPE_BF16 1

#define QLORA_ACCUM_DX 1 /* qlora_linear_bwd: dx += result instead of dx = result */
#define QLORA_ACCUM_DA 2 /* qlora_linear_bwd: da += result (gradient accumulation) */
#define QLORA_ACCUM_DB 4 /* qlora_linear_bwd: db += result */

/*
 * The quantised weight record (device pointers, caller-owned).
 *   codes        uint8 [n*k/2]  two 4-bit codes per byte; element 2i of the
 *                               row-major weight in the HIGH nibble of byte i.
 *   absmax_q     int8  [n*k/64] double-quantised block scale of each block of
 *                               64 consecutive row-major elements.
 *   absmax_step  f32   [ceil(n*k/64 / 256)] one step per group of 256 scales.
 *   absmax_mean  f32   [1]      per-tensor mean of the raw block scales.
 * Restored scale of block b: a' = (float)absmax_q[b] * absmax_step[b/256] + absmax_mean
 * (two float32 roundings); restored weight: bf16_rn(L[code] * a').
 */
typedef struct qlora_nf4_weight {
  uint8_t* codes;
  int8_t* absmax_q;
  float* absmax_step;
  float* absmax_mean;
  int64_t n;
  int64_t k;
} qlora_nf4_weight;

/* ----------------------------------------------------------------- quantisation */

/* Bytes of workspace qlora_nf4_quantize needs for an [n, k] weight. */
int qlora_nf4_quantize_workspace_bytes(int64_t n, int64_t k, size_t* bytes);

/*
 * NF4-quantise a row-major weight w [n, k] (float32 or bfloat16, w_dtype) into
 * `out` (whose n and k must equal the arguments).  Glossary "QLoRA", "How QLoRA
 * works": absmax of every 64 consecutive elements; code = index of the level
 * nearest to w / absmax (float32 division; ties to the lower index; an
 * all-zero block gives the zero level); then double quantisation of the
 * absmax array: mu = float32(RN64(exact sum of scales) / count), per group of
 * 256 scales step = max|a - mu| / 127 and q = clamp(rint((a - mu)/step), -127, 127)
 * (q = 0 where step == 0).  A non-finite weight latches QLORA_ERR_NONFINITE
 * (outputs then undefined).  Bit-exact against the definition.
 */
int qlora_nf4_quantize(const void* w, int w_dtype, int64_t n, int64_t k, const qlora_nf4_weight* out,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * qlora_nf4_quantize without a workspace argument, for callers that cannot
 * allocate device memory on the call path: plugins hosted by a framework that
 * owns all device memory through its own pool and forbids cudaMalloc/cudaFree
 * outside it, services with a memory budget fixed at start-up, and
 * latency-critical code where a cudaMalloc or cudaFree (which can synchronise
 * the device) is not acceptable.  The pages have no counterpart of this call;
 * it computes exactly what qlora_nf4_quantize computes (same kernels, same
 * bits), with the scratch taken from a fixed module-scope device array.
 *   - Limit: n * k <= 2^26 weights (1,048,576 absmax blocks; 4 MiB + 2.3 KiB of
 *     scratch, held on every device that has loaded the library's kernels,
 *     until exit).  Larger weights return QLORA_ERR_UNSUPPORTED before
 *     anything is launched.
 *   - Allocates nothing on the call path: no cudaMalloc, cudaFree or
 *     allocating library call.
 *   - When the scratch is reserved: under CUDA's default lazy module loading
 *     the library's device code, and with it the scratch, is loaded on a
 *     device by the first call that needs it -- the first call of this entry
 *     point on that device (which looks up the scratch address with
 *     cudaGetSymbolAddress, with that device current, and caches it) or of any
 *     other entry point that launches a kernel.  A caller whose memory budget
 *     is fixed at start-up should therefore make one call on each device at
 *     start-up (also before any stream capture), or run with
 *     CUDA_MODULE_LOADING=EAGER so the scratch is reserved when the CUDA
 *     context is created.
 *   - All calls on a device share the scratch.  Each call clears the parts
 *     that must start at zero and overwrites the rest, but calls whose kernels
 *     overlap on the GPU (different streams without ordering) race on it:
 *     order them on one stream.
 */
int qlora_nf4_quantize_noalloc(const void* w, int w_dtype, int64_t n, int64_t k, const qlora_nf4_weight* out,
                               void* stream);

/*
 * Dequantise the whole record to bfloat16 out [n, k] (glossary "QLoRA", "How
 * QLoRA works": restored weight = level * restored scale, in bfloat16).
 * Bit-exact against the definition in the record comment above.
 */
int qlora_nf4_dequantize(const qlora_nf4_weight* w, uint16_t* out, void* stream);

/* ----------------------------------------------------------------- merge / export */

/*
 * Merge the trained LoRA branch into the dequantised base:
 *   out bf16 [n, k] = bf16_rn( deq(W) + s * (B A) ),   s = alpha / r
 * (Day 25 notes "Fine-tuning and LoRA/QLoRA", section 2.6: W_merged = W0 + B A;
 * P1 tutorial "QLoRA: fine-tuning 7B on a 24 GB card", section 3.8, and glossary
 * "QLoRA", "Trade-offs": a 4-bit base is dequantised to 16 bits before the
 * merge, and re-quantised for serving -- pass `out` to qlora_nf4_quantize).
 *   lora_a bf16 [r, k], lora_b bf16 [n, r], 1 <= r <= 128.
 * Arithmetic (bit-exact against this definition): deq(W) as qlora_nf4_dequantize
 * gives it; (B A)[n, k] accumulated in float32 over j = 0 .. r-1 in that order,
 * one fused multiply-add per term (the bf16 products are exact); s * (B A)
 * rounded to float32, added to deq(W) in float32, rounded to bf16.
 */
int qlora_nf4_merge(const qlora_nf4_weight* w, const uint16_t* lora_a, const uint16_t* lora_b, int r, float alpha,
                    uint16_t* out, void* stream);

/*
 * Dense low-rank update in float32, the arithmetic step of the LoftQ
 * initialisation (P1 tutorial, section 3.10: alternate quantising the weight
 * minus the LoRA branch and fitting the branch to what quantisation lost):
 *   out f32 [n, k] = (W - deq(sub)) + coef * (B A)
 *   w      float32 or bfloat16 [n, k] (w_dtype), k % 64 == 0
 *   sub    NF4 record [n, k] subtracted from W, or NULL (nothing subtracted)
 *   lora_a bf16 [r, k], lora_b bf16 [n, r], 0 <= r <= 128 (r == 0: no B A
 *          term; the pointers may then be NULL)
 * Each float32 operation rounds once; B A is the same float32 FMA chain as in
 * qlora_nf4_merge.  With coef = -alpha / r it gives the weight LoftQ quantises;
 * with sub set and r == 0, the residual it factorises.
 */
int qlora_lowrank_update(const void* w, int w_dtype, int64_t n, int64_t k, const qlora_nf4_weight* sub,
                         const uint16_t* lora_a, const uint16_t* lora_b, int r, float coef, float* out, void* stream);

/* ----------------------------------------------------------------- the QLoRA linear */

/* Bytes of workspace qlora_linear_fwd needs for m tokens of an [n, k] weight with rank r. */
int qlora_linear_fwd_workspace_bytes(int64_t m, int64_t n, int64_t k, int r, size_t* bytes);

/*
 * Forward: Y = X deq(W)^T + s (X A^T) B^T with s = alpha / r (Day 25 notes,
 * sections 2.1 and 6.2; glossary "QLoRA", "How QLoRA works").
 *   x      bf16 [m, k]      input tokens
 *   lora_a bf16 [r, k]      LoRA A
 *   lora_b bf16 [n, r]      LoRA B
 *   y      bf16 [m, n]      output (overwritten)
 *   t_save f32  [m, r]      X A^T, written for the backward pass
 * The NF4 codes are decoded straight into tensor-core operands; no bf16 copy
 * of W is written to memory.  Accumulation is float32; s (X A^T) enters the
 * product rounded to bfloat16.  With 1 <= m <= 16 (and k <= 131072) the call
 * runs as a one-problem qlora_linear_fwd_grouped launch (the weight-streaming
 * decode kernel and its reading bf16(L[code]) * a', see there); it then uses
 * the first 256 bytes of the workspace as counters and zeroes them itself.
 */
int qlora_linear_fwd(const uint16_t* x, int64_t m, const qlora_nf4_weight* w, const uint16_t* lora_a,
                     const uint16_t* lora_b, int r, float alpha, uint16_t* y, float* t_save, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Bytes of workspace qlora_linear_bwd needs. */
int qlora_linear_bwd_workspace_bytes(int64_t m, int64_t n, int64_t k, int r, size_t* bytes);

/*
 * Backward of qlora_linear_fwd for upstream gradient dy bf16 [m, n]
 * (glossary "QLoRA", "How QLoRA works": gradients go through the dequantised
 * weight, only the LoRA matrices are updated -- there is no dW output):
 *   U  = dY B
 *   dx bf16 [m, k] = dY deq(W) + s U A
 *   da f32  [r, k] = s U^T X
 *   db f32  [n, r] = s dY^T T        (T = t_save from the forward)
 * flags: QLORA_ACCUM_DX / QLORA_ACCUM_DA / QLORA_ACCUM_DB add into the outputs.
 * s U and s T enter the tensor-core products rounded to bfloat16.
 */
int qlora_linear_bwd(const uint16_t* dy, const uint16_t* x, int64_t m, const qlora_nf4_weight* w,
                     const uint16_t* lora_a, const uint16_t* lora_b, int r, float alpha, const float* t_save,
                     uint16_t* dx, float* da, float* db, int flags, void* workspace, size_t workspace_bytes,
                     void* stream);

/* ----------------------------------------------------------------- LoRA dropout */

/*
 * Keep mask of LoRA dropout for an [m, k] branch input (k % 64 == 0): one bit
 * per element, bit e % 8 of byte e / 8 for element e = row * k + col (1 = kept),
 * m * k / 8 bytes.  Every page's LoRA configuration sets lora_dropout = 0.05
 * (P1 tutorial section 3.3; tbr8.org section 4; fedte.cc section 2).  Drawn by
 * Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3",
 * 2011): element e takes 32-bit word e % 4 of Philox(counter = (e / 4 low
 * word, e / 4 high word, offset low word, offset high word), key = (seed low
 * word, seed high word)) and is kept when that word >= floor(p * 2^32),
 * 0 <= p < 1.  A fresh (seed, offset) per step gives a fresh mask; the same
 * pair gives the same bits on every device.
 */
int qlora_dropout_mask(uint64_t seed, uint64_t offset, int64_t m, int64_t k, float p, uint8_t* mask, void* stream);

/*
 * qlora_linear_fwd with dropout on the LoRA branch input (inverted dropout: the
 * kept elements are scaled by 1 / (1 - p); the frozen path sees x itself):
 *   x_drop bf16 [m, k] = x * mask        (written; keep it for the backward)
 *   t_save f32  [m, r] = (x_drop A^T) / (1 - p)
 *   y      bf16 [m, n] = x deq(W)^T + s t_save B^T
 * mask as qlora_dropout_mask writes it; same workspace as qlora_linear_fwd.
 */
int qlora_linear_fwd_dropout(const uint16_t* x, int64_t m, const qlora_nf4_weight* w, const uint16_t* lora_a,
                             const uint16_t* lora_b, int r, float alpha, const uint8_t* mask, float p,
                             uint16_t* x_drop, uint16_t* y, float* t_save, void* workspace, size_t workspace_bytes,
                             void* stream);

/*
 * Backward of qlora_linear_fwd_dropout (the same mask, p, and the forward's
 * x_drop and t_save): U = dY B;
 *   dx = dY deq(W) + (s U A) * mask / (1 - p)
 *   da = s U^T x_drop / (1 - p),   db = s dY^T t_save
 * Flags and workspace as qlora_linear_bwd.  The LoRA term of dx goes through
 * the mask, so it is added to the frozen-path product after the GEMM (one more
 * rounding to bf16 than without dropout).
 */
int qlora_linear_bwd_dropout(const uint16_t* dy, const uint16_t* x_drop, int64_t m, const qlora_nf4_weight* w,
                             const uint16_t* lora_a, const uint16_t* lora_b, int r, float alpha, const uint8_t* mask,
                             float p, const float* t_save, uint16_t* dx, float* da, float* db, int flags,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * One small-token forward problem of a grouped call (host struct; the
 * pointers in it are device pointers, `w` points to a host record struct).
 */
typedef struct qlora_linear_problem {
  const uint16_t* x;           /* bf16 [m, k], 1 <= m <= 16 */
  int64_t m;
  const qlora_nf4_weight* w;   /* [n, k] */
  const uint16_t* lora_a;      /* bf16 [r, k] */
  const uint16_t* lora_b;      /* bf16 [n, r] */
  int r;                       /* 1 <= r <= 128 */
  float alpha;
  uint16_t* y;                 /* bf16 [m, n] (overwritten) */
  float* t_save;               /* f32 [m, r] = X A^T, or NULL */
} qlora_linear_problem;

/*
 * Bytes of workspace qlora_linear_fwd_grouped needs for this list on the
 * current device (the split of the weight stream over the SMs depends on the
 * device's SM count).
 */
int qlora_linear_fwd_grouped_workspace_bytes(const qlora_linear_problem* problems, int count, size_t* bytes);

/*
 * qlora_linear_fwd for a list of independent small-token problems (decode:
 * each matrix of a layer stack, or one decoder stage's q,k,v, applied to
 * 1..16 tokens), in ONE kernel launch per 128 problems.  The launch starts
 * while the preceding kernel of the stream still runs, pre-loads its weight
 * codes into L2 and waits for that kernel only before it reads anything the
 * stream wrote (x, the workspace), so consecutive calls keep HBM streaming.
 * Arithmetic: bf16 operands, float32 accumulation, s X A^T rounded to bf16 as
 * in qlora_linear_fwd; the weights enter as bf16(L[code]) with the block scale
 * a' applied in float32 to each 64-wide block's partial sum (within 2^-8 per
 * weight of the bf16_rn(L a') qlora_linear_fwd uses).  Each 16-row tile of y
 * is summed by one CTA in a fixed order, so every y is deterministic.
 * `problems` is a host array of `count` entries; 1 <= m <= 16, 1 <= r <= 128,
 * k <= 131072 (QLORA_ERR_UNSUPPORTED otherwise).  The weight codes are read
 * before the wait for the preceding kernel: a kernel that writes the weight
 * records must complete before the call (every kernel of this library that
 * writes a record does).
 * The workspace holds counters (X A^T slices published, tiles finished) and
 * the X A^T slice partials: it must be zero-filled
 * before its first use (cudaMemsetAsync once); every call returns them to zero,
 * so it may then be reused by later calls (and graph replays) ordered on the
 * same stream.  After a call that latched QLORA_ERR_TIMEOUT, zero it again.
 */
int qlora_linear_fwd_grouped(const qlora_linear_problem* problems, int count, void* workspace, size_t workspace_bytes,
                             void* stream);

/* ----------------------------------------------------------------- optimizer */

#define QLORA_ADAMW_PREFETCH 1 /* qlora_adamw_step: migrate managed state to the device before the update */

/* One trained tensor (a LoRA A or B) for qlora_adamw_step; device-accessible pointers. */
typedef struct qlora_adamw_tensor {
  float* master;        /* f32 [numel] weights, updated in place */
  uint16_t* param;      /* bf16 [numel] copy the linear reads (A or B), written; may be NULL */
  const float* grad;    /* f32 [numel] gradient (dA or dB of qlora_linear_bwd) */
  float* exp_avg;       /* f32 [numel] first moment, updated */
  float* exp_avg_sq;    /* f32 [numel] second moment, updated */
  int64_t numel;
} qlora_adamw_tensor;

/*
 * One AdamW step (decoupled weight decay; Loshchilov and Hutter 2019) on a list
 * of tensors, in one kernel launch per 240 tensors.  The pages train only the
 * LoRA matrices with a paged AdamW (P1 tutorial section 3.3, optim =
 * "paged_adamw_8bit"; tbr8.org section 5, "paged_adamw_32bit"; glossary
 * "QLoRA", "How QLoRA works": optimizer state in NVIDIA unified memory, paged
 * to CPU RAM during memory spikes).  This is the 32-bit variant: master
 * weights, exp_avg and exp_avg_sq in float32; they may live in memory from
 * cudaMallocManaged, which the driver pages between GPU and host on demand
 * (QLORA_ADAMW_PREFETCH migrates each managed range to the device on `stream`
 * before the update instead of faulting it in page by page).  The library
 * allocates nothing.  Per element, every float32 operation rounded once, in
 * this order (bit-exact against the definition):
 *   p = master * (1 - lr wd);  m = b1 m + (1 - b1) g;  v = b2 v + (1 - b2)(g g);
 *   p = p - (lr / (1 - b1^t)) * (m / (sqrt(v) / sqrt(1 - b2^t) + eps));
 *   master = p;  param = bf16_rn(p)
 * with 1 - lr wd, 1 - b1, 1 - b2, lr / (1 - b1^t) and sqrt(1 - b2^t) formed
 * in double precision and rounded to float32.  step t >= 1 (1 for the first
 * update); 0 <= b1, b2 < 1; eps > 0.  Tensors must not overlap.
 */
int qlora_adamw_step(const qlora_adamw_tensor* tensors, int count, float lr, float beta1, float beta2, float eps,
                     float weight_decay, int64_t step, int flags, void* stream);

/* ----------------------------------------------------------------- MLP glue */

/*
 * h = silu(g) * u elementwise on `count` bf16 values (count even, float32 math).
 * Not on the pages: the plain definition of the gate between the gate/up and
 * down projections of a Llama MLP block.
 */
int qlora_silu_mul_fwd(const uint16_t* g, const uint16_t* u, uint16_t* h, int64_t count, void* stream);

/* dg = dh * u * sigma(g) * (1 + g (1 - sigma(g))),  du = dh * silu(g). */
int qlora_silu_mul_bwd(const uint16_t* dh, const uint16_t* g, const uint16_t* u, uint16_t* dg, uint16_t* du,
                       int64_t count, void* stream);

/* ----------------------------------------------------------------- status and diagnostics */

/*
 * Synchronise `stream`, return and clear the latched device status of the
 * current device: QLORA_OK, QLORA_ERR_TIMEOUT, QLORA_ERR_NONFINITE, or
 * QLORA_ERR_CUDA if the synchronisation itself failed.
 */
int qlora_get_status(void* stream);

/* Static description of a return code. */
const char* qlora_strerror(int code);

/* Details of the last error returned on this host thread ("" if none). */
const char* qlora_last_error(void);

/*
 * Time limit of every bounded wait inside the kernels, in nanoseconds
 * (default 2e9).  A kernel whose wait expires latches QLORA_ERR_TIMEOUT,
 * releases its tensor memory and returns; the context stays usable.
 */
int qlora_set_wait_limit_ns(uint64_t ns);

/*
 * Launch one CTA that waits on an mbarrier no one arrives on, with limit
 * `wait_ns`.  The following qlora_get_status must return QLORA_ERR_TIMEOUT.
 * Exercises the timeout path without faulting or hanging the GPU.
 */
int qlora_selftest_wait_timeout(uint64_t wait_ns, void* stream);

/* Number of multiprocessors the kernels size their grids for (0 if no device). */
int qlora_device_sm_count(void);

/* ----------------------------------------------------------------- host <-> device copies */

/*
 * Moving a step's inputs and results between pinned host memory and the GPU.
 * Not on the pages: plumbing for feeding the linears from the host.
 *
 * qlora_copy_many copies `count` byte ranges, in stream order on `stream`:
 * each copy is cut into pieces of at least 2 MB, dealt round-robin over four
 * internal copy streams forked from `stream` (one cudaMemcpyAsync per piece)
 * and joined back before the call returns, so several copy engines share the
 * host link (one stream moves about 30 GB/s host-to-device on a B300's PCIe 6
 * x16 link, four about 50).  dst and src are any pointers the CUDA runtime
 * can address (device memory, pinned or registered host memory; pageable host
 * memory works but is not asynchronous); ranges must not overlap.  The caller
 * owns every buffer.  count == 0 is a no-op.  Errors: INVALID_ARGUMENT (NULL
 * list, or a NULL pointer with a non-zero size), CUDA (a copy could not be
 * issued).  Works inside a stream capture (the fork and join become graph edges).
 */
typedef struct {
  void* dst;
  const void* src;
  size_t bytes;
} qlora_copy;
int qlora_copy_many(const qlora_copy* copies, int count, void* stream);

/* ----------------------------------------------------------------- tracing */

/* Total number of kernels the entry points above have launched in this process. */
unsigned long long qlora_launch_count(void);

/*
 * While on, every kernel launch made by an entry point is bracketed by two
 * CUDA events on its stream (a few microseconds of host work per launch).
 * qlora_profile_collect() waits for the recorded events and adds their
 * elapsed times into per-launcher totals, read with qlora_profile_name /
 * _total_ms / _calls for i in [0, qlora_profile_collect()).  Names are the
 * launchers: "fwd_gemm", "bwd_dx_gemm", "lora_down", "lora_grads", ...
 */
int qlora_profile_enable(int on);
int qlora_profile_collect(void);
const char* qlora_profile_name(int i);
double qlora_profile_total_ms(int i);
long long qlora_profile_calls(int i);
int qlora_profile_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_NF4_H_ */
