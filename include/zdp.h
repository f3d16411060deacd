/*
 * zdp.h -- C ABI of libzdp, the ZeRO synchronisation-and-update step on one
 * GPU.  P logical data-parallel ranks keep their gradients and parameter
 * replicas as separate buffers in one GPU's memory.  One step
 *   1. reduce-scatters the P gradients: element i is owned by rank
 *      r = i / S, S = ceil(n / P), and summed in fp32 in ring order,
 *      starting with rank (r+1) mod P and ending with rank r, then multiplied
 *      by `scale`;
 *   2. applies AdamW to the owner's shard of the fp32 master weight, first
 *      moment m and second moment v;
 *   3. rounds the new master weight to bf16 (nearest, ties to even) and
 *   4. all-gathers it into every rank's replica.
 *
 * Sources, by page title and section:
 *  - Fudan MLSys ch. 9 "Distributed training and data parallelism":
 *    9.2.2 Adam (moment updates, bias correction, epsilon outside the
 *    square root); 9.3.6 ring all-reduce = ring reduce-scatter (P-1 steps,
 *    each adding the received partial sum to the local chunk) + ring
 *    all-gather (P-1 steps, overwrite); 9.4.2 ZeRO-1/2 step
 *    (reduce-scatter gradients, update the own shard, all-gather params).
 *  - CS336 Lecture 7 notes "Parallelism I": 3.4 all-reduce = reduce-scatter
 *    + all-gather; 4.2 ring schedule; 6.2 gradient averaging as SUM then
 *    divide by world size; 7 the 16 bytes/parameter mixed-precision state
 *    (bf16 param, bf16 grad, fp32 master, m, v); 8.1 FlatZeRO1 (flatten all
 *    parameters, split into P equal segments); 11 exercise 1(e) (zero
 *    padding to a multiple of P).
 *  - "Must-know: communication cost of LLM training" interview guide, 1.4
 *    item 6: after a reduce-scatter GPU r holds reduced chunk r.
 * The pages name AdamW without writing its decay term; this library uses
 * decoupled decay on the pre-update weight:
 *   w <- w - (lr*wd)*w - lr * (m_hat / (sqrt(v_hat) + eps)).
 *
 * Conventions for every call:
 *  - The caller owns all memory.  No call allocates or frees device or host
 *    memory.  Device pointers are plain CUDA device addresses (e.g. a torch
 *    tensor's data_ptr()).  "Host array of P device pointers" means a
 *    host-memory array whose entries are device addresses.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream) and never synchronise.
 *  - Return value: ZDP_OK, or ZDP_ERR_INVALID when an argument check fails
 *    (detected on the host before anything is enqueued), or ZDP_ERR_CUDA when
 *    a CUDA call fails.  zdp_last_error() then returns a message (per host
 *    thread, valid until the thread's next call).
 *  - Element counts are int64.  P is 1..ZDP_MAX_P.
 *  - A non-finite reduced gradient is data, not an error: it is reported
 *    through the optional device overflow word.
 *  - Any 2-byte (bf16/fp16) or 4-byte (fp32) aligned pointer is accepted.
 *    When every buffer's element 0 sits on a 16-byte boundary (torch's
 *    allocations do) the kernels move 16 bytes per access; otherwise a
 *    slower one-element-per-access kernel runs, with identical results.
 *  - Output buffers must not overlap inputs or each other; overlapping
 *    ranges are rejected with ZDP_ERR_INVALID.
 */
#ifndef ZDP_H
#define ZDP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zdp_dtype {
  ZDP_BF16 = 0, /* bfloat16 gradients */
  ZDP_FP16 = 1, /* IEEE binary16 gradients (loss-scaled training) */
  ZDP_F32 = 2   /* fp32 (input of zdp_quantize_blocks only) */
} zdp_dtype;

/* Storage of the AdamW moments m and v.  ZDP_MOMENTS_BF16 keeps everything
 * except the fp32 master weight in bf16, 12 bytes of state per parameter
 * (CS336 Lecture 7 notes, 8.4): the moments are widened exactly on load,
 * updated in fp32 (the update uses these fp32 values), and rounded to
 * nearest even when stored. */
typedef enum zdp_moment_dtype {
  ZDP_MOMENTS_F32 = 0,
  ZDP_MOMENTS_BF16 = 1
} zdp_moment_dtype;

enum {
  ZDP_OK = 0,
  ZDP_ERR_INVALID = -1,
  ZDP_ERR_CUDA = -2,
  ZDP_MAX_P = 64
};

/* Bits of the d_overflow word. */
#define ZDP_FLAG_OVERFLOW 1 /* some reduced gradient was not finite */
#define ZDP_FLAG_TIMEOUT 2  /* the single-pass checked step's grid barrier timed out.  The
                               range's master, m, v and replicas are then unspecified (some
                               blocks may have written their part, others not): the caller
                               must restore them, e.g. from a copy, before the next step
                               (see zdp_step) */

/* Library version, e.g. 100 for 0.1.0. */
int zdp_version(void);

/* Shard size S = ceil(n / P): rank r owns flat elements [r*S, (r+1)*S);
 * elements at or beyond n are zero padding (CS336 Lecture 7 notes,
 * exercise 1(e); FlatZeRO1 in 8.1).  Returns -1 if n < 1 or P is outside
 * 1..ZDP_MAX_P.  Pure host function. */
int64_t zdp_shard_size(int64_t n, int P);

/* Reduce-scatter (step 1 alone).
 *   grads      host array of P device pointers; grads[q] holds rank q's n
 *              gradients (bf16 or fp16 per gdt).
 *   shards     device fp32 output of P*S elements: shards[i] is the ring-order
 *              sum of element i times `scale` for i < n, and 0.0 for the
 *              padding i in [n, P*S).  Rank r's shard is shards + r*S.
 *   d_overflow nullable device int32; OR-ed with 1 if any shards[i] is not
 *              finite (never cleared by the call).
 *   d_sumsq    nullable device double; the fp64 sum of shards[i]^2 is added
 *              to it (never cleared by the call).
 * Source: Fudan MLSys ch. 9, 9.3.6 (reduce-scatter phase of the ring);
 * the interview guide 1.4 item 6 (rank r keeps chunk r). */
int zdp_reduce_scatter(const void* const* grads, int gdt, float* shards, int64_t n, int P,
                       float scale, int32_t* d_overflow, double* d_sumsq, void* stream);

/* AdamW on one shard (step 2 alone), elementwise over `count` elements:
 *   m <- b1*m + (1-b1)*g;  v <- b2*v + (1-b2)*g*g;
 *   u  = (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + eps);
 *   w <- w - (lr*wd)*w;  w <- w - lr*u.
 * Every operation is one IEEE fp32 operation rounded to nearest (no fused
 * multiply-add); 1-b^t is evaluated in double and rounded to fp32.
 *   master, m, v  device fp32, count elements each, updated in place.
 *   grad_shard    device fp32, count elements (e.g. a zdp_reduce_scatter shard).
 *   t             step number, >= 1.
 * Source: Fudan MLSys ch. 9, 9.2.2. */
int zdp_adamw_shard(float* master, float* m, float* v, const float* grad_shard, int64_t count,
                    float lr, float b1, float b2, float eps, float wd, int t, void* stream);

/* All-gather of the updated parameters (steps 3 and 4 alone): for i < n and
 * every rank q, replicas[q][i] = bf16(master[i]), rounded to nearest even.
 *   master    device fp32, at least n elements (the concatenated shards).
 *   replicas  host array of P device pointers, n bf16 (uint16) each.
 * Source: Fudan MLSys ch. 9, 9.3.6 (all-gather phase: overwrite only);
 * CS336 Lecture 7 notes 8.1 step 4 (all-gather the parameters). */
int zdp_all_gather(const float* master, uint16_t* const* replicas, int64_t n, int P,
                   void* stream);

/* Arguments of the fused step. */
typedef struct zdp_step_args {
  const void* const* grads;   /* host array of P device pointers; grads[q][j] is rank
                                 q's gradient of global element off+j, j < len */
  int gdt;                    /* zdp_dtype of the gradients */
  float* master;              /* device fp32, >= n elements, indexed by global element */
  void* m;                    /* device, >= n elements: fp32, or bf16 per moment_dtype */
  void* v;                    /* device, >= n elements: fp32, or bf16 per moment_dtype */
  uint16_t* const* replicas;  /* host array of P device pointers, >= n bf16 each,
                                 indexed by global element */
  int64_t n;                  /* model size; fixes S = ceil(n/P) and so the owners */
  int64_t off;                /* first global element this call processes */
  int64_t len;                /* number of elements this call processes (may be 0) */
  int P;                      /* logical ranks, 1..ZDP_MAX_P */
  float scale;                /* multiplies the ring sum, e.g. 1/P or 1/(P*loss_scale) */
  float lr, b1, b2, eps, wd;  /* AdamW hyper-parameters */
  int t;                      /* AdamW step number, >= 1 */
  int64_t bucket_elems;       /* > 0: walk [off, off+len) in buckets of this many
                                 elements (one launch each); 0: whole range at once */
  int check_overflow;         /* nonzero: if any reduced gradient in the range is not
                                 finite, write nothing to master/m/v/replicas */
  int32_t* d_overflow;        /* nullable device int32, OR-ed with ZDP_FLAG_OVERFLOW (1)
                                 on a non-finite reduced gradient in the range, and
                                 with ZDP_FLAG_TIMEOUT (2) as zdp_step describes */
  double* d_sumsq;            /* nullable device double; the fp64 sum of squares of
                                 the reduced gradients of the range is added */
  void* workspace;            /* device scratch for check_overflow (else unused), at
                                 least zdp_step_workspace_bytes() bytes, 16-B aligned */
  size_t workspace_bytes;
  int moment_dtype;           /* zdp_moment_dtype of m and v (0: fp32) */
} zdp_step_args;

/* Scratch bytes zdp_step needs for these arguments: 0 without
 * check_overflow, else 4*len rounded up to 256, plus 256. */
size_t zdp_step_workspace_bytes(const zdp_step_args* args);

/* The fused step over global elements [off, off+len): reduce-scatter, AdamW,
 * bf16 cast and all-gather in one pass over memory (CS336 Lecture 7 notes
 * 8.1, FlatZeRO1; Fudan MLSys ch. 9, 9.4.2, ZeRO-1/2 step).  Ownership and
 * summation order depend only on the global index and n, never on off, len
 * or bucket_elems, so any split of [0, n) into calls or buckets gives
 * bit-identical results.
 * With check_overflow the call makes two passes: the first stores the
 * reduced gradients in the workspace and raises a device flag on any
 * non-finite value; the second, skipped on the device when the flag is set,
 * applies AdamW and the all-gather.  When the 16-byte vector path applies, P
 * is 1..8, 16, 32 or 64, and the range's reduced gradients fit in the
 * registers of one resident wave (about 2 million elements on a GB300), it
 * instead makes one cooperative launch that keeps them in registers across a
 * grid barrier (same results, 8 fewer bytes per element and one launch
 * instead of two).  If the device cannot run that launch (e.g. fewer SMs are
 * available to the process than the device reports), the call falls back to
 * the two passes.  That barrier waits at most ZDP_COOP_TIMEOUT_NS
 * nanoseconds (environment variable, default 1e9); a block that gives up
 * writes nothing of its part of the range and ORs ZDP_FLAG_TIMEOUT into
 * *d_overflow, while blocks whose wait ended in time go on and write theirs.
 * So after a timeout the range's master, m, v and replicas are unspecified,
 * a mix of old and new values, whatever the overflow bit says: the caller
 * must restore them (from a copy taken before the call, or a checkpoint) and
 * may rerun the step.  The barrier only times out if the GPU is preempted or
 * shared so heavily that the resident blocks stop making progress.  Environment
 * variable ZDP_COOP=0 selects the two-pass form always, and
 * ZDP_TEST_COOP_EXTRA_ARRIVALS=k (tests only) makes the barrier wait for k
 * arrivals that never come, and ZDP_TEST_COOP_OVERSIZE=k (tests only) asks
 * for a cooperative grid k blocks larger than one resident wave, which the
 * runtime refuses, so that the two-pass fallback runs.  The skip decision
 * covers this call's range only; a caller streaming one step through several
 * calls and wanting a step-wide skip must check every range first (e.g. with
 * zdp_reduce_scatter into a scratch buffer).  A skipped step leaves t to the
 * caller: do not advance it. */
int zdp_step(const zdp_step_args* args, void* stream);

/* The same step as zdp_step, run as the literal ring schedule of the pages
 * instead of one fused pass, for measuring what the fused pass saves.
 * Reduce-scatter: P-1 launches; at step s every rank i adds its own chunk
 * (i-s-1) mod P to the fp32 partial sum received from rank i-1 (Fudan MLSys
 * ch. 9, 9.3.6; CS336 Lecture 7 notes 4.2, in the labelling where rank r
 * finishes chunk r).  Then one launch: the owner's last add, scale, AdamW and
 * the bf16 write of the owner's chunk of its own replica.  All-gather: P-1
 * launches, step s copying chunk (i-s) mod P of replica i into replica i+1.
 * The partial sums travel through `workspace` (2*P*S fp32 "messages",
 * zdp_step_ring_workspace_bytes(args) bytes, 16-byte aligned).
 * Results are bit-identical to zdp_step (same additions in the same order).
 * The call covers the whole model: off = 0, len = n, bucket_elems = 0,
 * check_overflow = 0 and fp32 moments are required (ZDP_ERR_INVALID
 * otherwise); d_overflow and
 * d_sumsq work as for zdp_step.  With bf16 gradients it moves about
 * (14P + 14) bytes of HBM traffic per parameter (each of the P-2 middle
 * reduce-scatter steps reads and writes the fp32 messages), against
 * (4P + 24) for zdp_step. */
size_t zdp_step_ring_workspace_bytes(const zdp_step_args* args);
int zdp_step_ring(const zdp_step_args* args, void* stream);

/* ZeRO++ (Fudan MLSys ch. 9, 9.4.3: the weights are converted to INT8
 * before the all-gather and dequantized after it; gradients are quantized
 * block-wise for the reduce-scatter).  Blocks are ZDP_QBLOCK = 256
 * consecutive elements, global element i in block i / 256.  A block's scale
 * is max|x| / 127 (fp32), q = x / scale rounded half to even and clamped to
 * [-127, 127]; an all-zero block has scale 0; x is recovered as q * scale in
 * fp32.  A block holding a NaN has a NaN scale and one holding an infinity
 * (and no NaN) an infinite scale; a NaN quotient x / scale gives q = -127.
 * Such a block dequantizes to non-finite values, so a non-finite gradient
 * that reaches the quantized reduce-scatter raises the overflow flag. */
#define ZDP_QBLOCK 256

/* Quantize n values (xdt: ZDP_BF16, ZDP_FP16 or ZDP_F32) into q (n int8)
 * and scales (ceil(n/256) fp32, block b covering [256b, 256b+256)): the
 * producer's side of the quantized reduce-scatter. */
int zdp_quantize_blocks(const void* x, int xdt, int64_t n, int8_t* q, float* scales,
                        void* stream);

/* out[i] = bf16(q[i] * scales[i / 256]), rounded to nearest even: the
 * receiver's side of the quantized all-gather. */
int zdp_dequantize_blocks(const int8_t* q, const float* scales, int64_t n, uint16_t* out,
                          void* stream);

/* Arguments of the ZeRO++ step: as zdp_step_args, with int8 block-quantized
 * gradients in and int8 block-quantized replicas out. */
typedef struct zdp_zpp_args {
  const int8_t* const* grads;      /* host array of P device pointers; grads[q][j] is rank
                                      q's int8 gradient of global element off+j, j < len */
  const float* const* grad_scales; /* host array of P device pointers; grad_scales[q][b] is
                                      the scale of global block off/256 + b */
  float* master;                   /* device fp32, >= n elements, global index */
  void* m;                         /* device, >= n elements, fp32 or bf16 per moment_dtype */
  void* v;
  int moment_dtype;
  int8_t* const* replicas;         /* host array of P device pointers, >= n int8 each;
                                      global index */
  float* const* replica_scales;    /* host array of P device pointers, >= ceil(n/256) fp32
                                      each; global block index */
  int64_t n, off, len;             /* off a multiple of 256; off+len a multiple of 256 or n */
  int P;
  float scale, lr, b1, b2, eps, wd;
  int t;
  int32_t* d_overflow;             /* nullable, as in zdp_step_args */
  double* d_sumsq;                 /* nullable, as in zdp_step_args */
} zdp_zpp_args;

/* The step with quantized communication: element i's reduced gradient is
 * the ring-order fp32 sum (as in zdp_step) of the P ranks' dequantized int8
 * gradients, times scale; AdamW as in zdp_step; the new bf16 parameters are
 * block-quantized once and the int8 values and scales written to every
 * rank's replica.  HBM traffic per parameter: P int8 gradient reads, the
 * state (24 bytes with fp32 moments, 16 with bf16), P int8 replica writes,
 * and one fp32 scale per 256 elements per rank each way: 2P + 24 + P/32
 * bytes with fp32 moments (40.25 at P = 8, against 56 for zdp_step).  All
 * buffers must have element 0 on a 16-byte boundary (the scale arrays on a
 * 4-byte one); no overflow skip (the flag is reported). */
int zdp_step_zpp(const zdp_zpp_args* args, void* stream);

/* Largest `len` zdp_step_noalloc accepts (16,777,216 elements). */
#define ZDP_NOALLOC_MAX_LEN 16777216LL

/* The overflow-checked fused step (zdp_step with check_overflow = 1) for
 * callers that cannot allocate device memory.  The pages have no counterpart
 * to this call; it exists for callers such as a plug-in living inside a
 * framework whose caching allocator owns the device memory (a raw cudaMalloc
 * would bypass its accounting, or fail once the pool holds the free memory),
 * or a step loop that must not call cudaMalloc/cudaFree because they
 * synchronise the device.
 *   args  as for zdp_step; check_overflow, workspace and workspace_bytes are
 *         ignored.  The call runs the overflow-checked step in whichever form
 *         zdp_step picks for the range (the single cooperative launch or the
 *         two passes); both forms keep their scratch (the flag and barrier
 *         words, and the two-pass form's reduced gradients) in a static device
 *         array inside libzdp of 64 MiB + 512 B, which every GPU that loads the
 *         library holds until the process exits.
 *   Returns ZDP_ERR_INVALID (nothing enqueued) when args->len exceeds
 *   ZDP_NOALLOC_MAX_LEN; split longer ranges into several calls.
 * It calls no allocating routine.  Its first call in a CUDA context (normally
 * the first on a device) looks up the scratch's device address in that context
 * with cudaGetSymbolAddress, which may load the library's module there; make
 * that first call before any stream capture.  Later calls reuse the address
 * found for the current context.  Every call in a context uses the same
 * scratch, which keeps the last call's contents (the call clears its flag and
 * barrier words itself): calls that may run at the same time on the GPU, e.g.
 * on two streams without an ordering between them, race on it. */
int zdp_step_noalloc(const zdp_step_args* args, void* stream);

/* A plain device-to-device copy of `bytes` bytes with 16-byte streaming
 * loads and stores (ld/st.global.cs) on a persistent grid of 128-thread
 * blocks: the access pattern of the step's kernels with no arithmetic.  The
 * pages have no counterpart; it measures the copy ceiling the step is held
 * against.
 *   dst, src  device pointers, both 16-byte aligned, not overlapping.
 *   bytes     a non-negative multiple of 16 (0: nothing is enqueued).
 * Returns ZDP_ERR_INVALID (nothing enqueued) for a NULL pointer, a size or
 * alignment outside these rules, or overlapping ranges. */
int zdp_copy(void* dst, const void* src, int64_t bytes, void* stream);

/* Message for the last non-OK return on this host thread ("" if none). */
const char* zdp_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ZDP_H */
