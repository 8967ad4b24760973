/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed mixture-of-experts FFN with
 * block-scaled FP4 experts.
 *
 * The operation is one routed-MoE feed-forward layer as the pages on
 * streaming experts describe it: a router picks the top-k experts of a token
 * ("Running a 133 GB MoE model on an 8 GB GPU at 11 tokens/s by streaming
 * experts from NVMe", section "Why this model": top-10 of 512; "Running the
 * 510 GB DeepSeek-V4.1-Flash on an 8 GB GPU, and three bugs that never raise
 * an error", section "Bytes per token decide everything": 6 of 384); every
 * selected expert is one contiguous record gate | up | down | gate_scale |
 * up_scale | down_scale of FP4 (e2m1) codes with block scales (first page,
 * section "The engine", item 1); the expert computes SwiGLU
 * down(silu(gate x) * up x) (first page, "The engine", item 4); the outputs
 * are summed with the router weights.
 *
 * Conventions shared by every entry point:
 *  - All data pointers are DEVICE pointers owned by the caller, unless a
 *    comment says otherwise.  The library keeps no state between calls and
 *    allocates no memory.
 *  - BF16 tensors are passed as uint16_t bit patterns.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is asynchronous on that stream.
 *  - The return value is a moe_status: host-side argument checks and launch
 *    errors only.  Errors found while a kernel runs (a bad expert index, a
 *    NULL or misaligned record, a wait that ran out) are OR-ed into the
 *    optional device word `dev_status` (MOE_DEV_* bits); the kernel skips
 *    the bad item, never traps, and the caller reads the word after its own
 *    synchronisation.
 *  - Matrices are row-major [out x in] with the input dimension K contiguous:
 *    gate and up are [I x H], down is [H x I].
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* NULL pointer, negative or zero size, k > E ... */
  MOE_ERR_ALIGNMENT = 2,           /* a pointer is not 16-byte aligned */
  MOE_ERR_UNSUPPORTED = 3,         /* shape outside what the kernels handle */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the *_workspace() size */
  MOE_ERR_CUDA = 5                 /* a CUDA launch or runtime call failed */
} moe_status;

/* Record formats. */
enum {
  MOE_FMT_NVFP4 = 0, /* e2m1 codes + one FP8 E4M3 scale per 16 elements */
  MOE_FMT_MXFP4 = 1  /* e2m1 codes + one UE8M0 scale (2^(s-127)) per 32 elements */
};

/* Bits of the device status word. */
enum {
  MOE_DEV_NULL_EXPERT = 1, /* a selected expert's record pointer was NULL */
  MOE_DEV_MISALIGNED = 2,  /* a selected expert's record was not 16-byte aligned */
  MOE_DEV_BAD_INDEX = 4,   /* an expert index was outside [0, E) */
  MOE_DEV_TIMEOUT = 8,     /* a bounded wait inside a kernel gave up */
  MOE_DEV_FP16_RANGE = 16  /* prompt path, NVFP4: an activation's magnitude is >= 65520 */
};

/* Expert shape: hidden size H, intermediate size I, record format.
 * Supported: H and I multiples of 64, H <= 16384, I <= 8192. */
typedef struct {
  int32_t hidden;
  int32_t inter;
  int32_t format;
} moe_expert_shape;

/* Byte size of one expert record (first page, "The engine", item 1: one
 * 2,764,800-byte block for H=2560, I=640, NVFP4; second page, "The
 * approach": 17.7 MB of codes + 1.1 MB of scales for the DeepSeek shape).
 * Layout, all parts back to back, no padding:
 *   gate codes [I x H/2] | up codes [I x H/2] | down codes [H x I/2] |
 *   gate scales [I x H/G] | up scales [I x H/G] | down scales [H x I/G]
 * G = 16 (NVFP4) or 32 (MXFP4).  Codes hold two elements per byte, element
 * 2i in the low nibble.  Returns 0 for an unsupported shape. */
size_t moe_expert_record_bytes(moe_expert_shape s);

/* Byte offsets of the six parts plus the total, written to offsets[0..6]
 * (host array) in the order gate, up, down, gate_s, up_s, down_s, total. */
int moe_expert_record_offsets(moe_expert_shape s, size_t* offsets);

/* Quantise one expert from FP32 and pack its record (first page, "The
 * engine", item 1: the repacked one-block-per-expert format).
 * gate [I x H], up [I x H], down [H x I]: FP32 device arrays.
 * record: device buffer of moe_expert_record_bytes(s) bytes, 16-B aligned.
 * NVFP4 block of 16: s = E4M3_rn_satfinite(amax / 6) (FP32 divide); if the
 * decoded s is 0 every code is +0, else code = e2m1_rn_satfinite(x / s).
 * MXFP4 block of 32: s = clamp(E + 127, 0, 254) for the smallest E with
 * 6 * 2^E >= amax (s = 0 when amax = 0); code = e2m1_rn_satfinite(x * 2^(127-s)).
 * Round to nearest, ties to even; the sign of zero results is kept. */
int fp4_pack_expert(const float* gate, const float* up, const float* down,
                    moe_expert_shape s, void* record, void* stream);

/* Router: logits, top-k and renormalised softmax weights (first page, "Why
 * this model": top-10 routing; "Where the time actually goes": the router's
 * answer gates the expert work).
 * x_bf16 [T x H], wr_bf16 [E x H]: BF16, 16-B aligned, H % 8 == 0.
 * bias [E] FP32 or NULL.
 * logits [T x E] FP32 output (required): logit[t,e] = sum_h x[t,h] W_r[e,h]
 *   (+ bias[e]) summed in FP32 in a fixed order: the K axis is cut into
 *   chunks of 8; chunk c goes to slot c mod 32; each slot sums its chunks in
 *   ascending order from +0; the 32 slots are combined pairwise, slot i with
 *   slot i xor d for d = 16, 8, 4, 2, 1; the bias is added last.
 * idx [T x k] int32 output: the k largest logits, larger first, ties to the
 *   lower expert index, NaN last.
 * weights [T x k] FP32 output: exp(l_j - l_0) / sum_i exp(l_i - l_0) over
 *   the selected k (sums to 1).
 * Limits: 1 <= k <= min(E, 32), E <= 1024. */
int moe_router_topk(const uint16_t* x_bf16, const uint16_t* wr_bf16, const float* bias,
                    int T, int H, int E, int k,
                    int32_t* idx, float* weights, float* logits, void* stream);

/* Layer chaining for stacked decode: x[t] = BF16(y[t] * r), r = 1 /
 * sqrt(mean(y[t]^2) + eps), no learnable weight.  FP32 in one fixed order so
 * the result is reproducible bit for bit: thread i of 256 sums y[i + 256 m]^2
 * for m ascending (square rounded, then added), a pairwise tree adds partial
 * i + w into partial i for w = 128, 64, ..., 1, mean = sum / H, r uses IEEE
 * sqrt and divide, and y * r is rounded once to BF16 (ties to even).  eps is
 * rounded to FP32.
 * y [T x H] FP32 input, x_bf16 [T x H] output. */
int moe_rmsnorm_bf16(const float* y, int T, int H, double eps, uint16_t* x_bf16,
                     void* stream);

/* Layer chaining fused with the router, for stacked decode: x = RMS chaining
 * of y_prev exactly as moe_rmsnorm_bf16 computes it (written to x_out), then
 * moe_router_topk on that x.  Same outputs, same limits; when x takes at
 * most 40 KB (T*H*2 bytes) it is two launches: the logits on every SM (W_r
 * rows pulled into L2 before the wait on the previous kernel), then the
 * top-k. */
int moe_rmsnorm_router_topk(const float* y_prev, int T, int H, double eps, uint16_t* x_out,
                            const uint16_t* wr_bf16, const float* bias, int E, int k,
                            int32_t* idx, float* weights, float* logits, void* stream);

/* Workspace bytes moe_experts_decode needs for T tokens, k experts each:
 * a 16,640-byte header of counters, then the logits the CTAs of a one-shot
 * launch exchange (1024 per token, each an 8-byte word of the value and a
 * per-layer tag), then the FP32 SwiGLU intermediate [T*k][I] (the other
 * decode paths keep theirs right after the header).  Zero-fill it before
 * its first use.  Every call that completes
 * leaves the counters in a state the next call accepts, so one zeroed
 * workspace serves any number of calls, of any shape, on one stream; calls
 * that overlap in time need separate workspaces.  After a call that reported
 * MOE_DEV_TIMEOUT, zero it again.  For diagnosis, the 64-bit word at byte
 * 192 of the workspace then holds the first wait that gave up since the
 * zero-fill: site << 56 | (layer + 1) << 32 | CTA index, with site 1 the
 * router rows' copy, 2 the gate/up scales, 3 a gate/up piece, 4 the down
 * rows, 5 and 6 the two grid barriers of a layer, 7 the barrier between
 * layers (moe_decode_stack), 8 the copy warp's own wait. */
size_t moe_experts_decode_workspace(int T, int k, moe_expert_shape s);

/* Decode path: the experts of T tokens (T*k small, GEMV shaped), HBM bound
 * (first page, "The engine", item 4: the single-token NVFP4 SwiGLU expert
 * kernel).  Small calls (the selected rows fit in shared memory) run one
 * persistent kernel that copies every row at entry; up to T*k = 512 pairs a
 * persistent kernel streams the rows through a shared-memory ring; both have
 * a grid barrier between gate/up and down.  Larger calls use two kernels.
 * Results are bit-identical between repeated calls.
 * x_bf16 [T x H]; idx, weights [T x k] as moe_router_topk writes them.
 * expert_ptrs: device array of E device pointers, one record per expert;
 *   entries may point anywhere (arbitrary slots), 16-B aligned; an entry may
 *   be NULL if that expert is never selected.
 * y [T x H] FP32 output, overwritten:
 *   y[t] = sum_j weights[t,j] * down_e(silu(gate_e x_t) * up_e x_t),
 *   e = idx[t,j], with FP32 accumulation and an FP32 SwiGLU intermediate,
 *   summed in a fixed order (bit-reproducible).
 * workspace: device scratch of at least moe_experts_decode_workspace() bytes.
 * dev_status: device int32 or NULL; MOE_DEV_* bits are OR-ed into it.
 * Limits: T*k <= 4096, k*I <= 49152.
 * Residency: the one-shot and ring kernels run one CTA per SM with grid-wide
 * barriers, so all of their CTAs must be resident at once.  The library
 * checks on the host that one CTA fits on an SM (else MOE_ERR_CUDA).  The
 * launches are not cooperative (that would add host time to every launch),
 * so kernels of other streams, processes (MPS) or green contexts that hold
 * SMs for the whole call can keep CTAs out: the barrier waits then run out
 * (2 s) with MOE_DEV_TIMEOUT and NaN outputs rather than hang.  Do not run
 * such persistent kernels concurrently with this call. */
int moe_experts_decode(const uint16_t* x_bf16, const int32_t* idx, const float* weights,
                       int T, int k, const void* const* expert_ptrs, int E,
                       moe_expert_shape s, float* y, void* workspace, size_t ws_bytes,
                       int32_t* dev_status, void* stream);

/* Decode from a host-memory expert tier (first page, "The engine", items 1-2:
 * the experts live in host RAM and only the selected ones travel to the GPU
 * each token).  Same arguments, output and bits as moe_experts_decode's
 * two-kernel path, but every record byte is read with plain 16-byte loads,
 * so expert_ptrs may point into host memory that the device can address:
 * pinned host memory on a unified-address system, or the Grace CPU's memory
 * that a GB300 reaches over NVLink-C2C.  Records in HBM work too (then it is
 * simply the two-kernel path).  The records must not change while the call
 * runs.  Same workspace rules and limits as moe_experts_decode. */
int moe_experts_decode_host(const uint16_t* x_bf16, const int32_t* idx, const float* weights,
                            int T, int k, const void* const* expert_ptrs, int E,
                            moe_expert_shape s, float* y, void* workspace, size_t ws_bytes,
                            int32_t* dev_status, void* stream);

/* One decode layer in one launch (first page, "The engine", item 4, and
 * "Where the time actually goes": the expert work of a layer waits on the
 * router's answer, so router and experts share the launch and no index
 * leaves the device).  Computes exactly what moe_rmsnorm_router_topk (or
 * moe_router_topk when x_bf16 is given) followed by moe_experts_decode
 * compute, with the same outputs bit for bit:
 *  - exactly one of x_bf16 [T x H] (this layer's input) and y_prev [T x H]
 *    FP32 (the previous layer's output, RMS-chained with eps into x_out,
 *    which is then required) is non-NULL; x_out may be NULL with x_bf16;
 *  - logits [T x E], idx / weights [T x k] as the router entries write them;
 *  - y [T x H] as moe_experts_decode writes it; y may be the same buffer as
 *    y_prev (every read of y_prev precedes every write of y).
 * H = s.hidden; expert_ptrs holds E records; bias may be NULL.  The
 * workspace is moe_experts_decode's (same size, same zero-fill rule).
 * wr_bf16 and expert_ptrs are read as soon as the launch starts, before it
 * waits for the previous kernel on the stream (programmatic dependent
 * launch): they must not be written by a kernel that lets its dependents
 * start before it ends.
 * Shapes the one-shot expert pass does not cover (T*k > 64, or a per-SM
 * share larger than shared memory) return MOE_ERR_UNSUPPORTED: use the two
 * calls for those.  The residency requirement of moe_experts_decode (all CTAs
 * of the grid-barrier kernel resident at once) applies. */
int moe_decode_layer(const uint16_t* x_bf16, const float* y_prev, int T, double eps, uint16_t* x_out,
                     const uint16_t* wr_bf16, const float* bias, int E, int k, int32_t* idx,
                     float* weights, float* logits, const void* const* expert_ptrs,
                     moe_expert_shape s, float* y, void* workspace, size_t ws_bytes,
                     int32_t* dev_status, void* stream);

/* A whole decode stack in one launch (first page, "Why this model": 48
 * layers in a row, each routing the previous layer's output; "Where the time
 * actually goes": the per-layer issue overhead).  Computes exactly what
 * `layers` calls of moe_decode_layer compute -- layer 0 with x_bf16 = x0, each
 * later layer with y_prev = y (RMS-chained with eps) -- with the same bits,
 * in one persistent kernel whose layers are separated by grid barriers
 * instead of launch boundaries:
 *  - wr_bf16 [layers x E x H] BF16, bias [layers x E] FP32 or NULL,
 *    expert_ptrs [layers x E] (device): one block per layer, back to back;
 *  - idx, weights [layers x T x k]: each layer's routing;
 *  - logits [T x E]: scratch, the last layer's logits at the end;
 *  - x_out [T x H] (may be NULL): the last layer's input;
 *  - y [T x H]: the last layer's output (each layer's output in turn).
 * Same limits, workspace rules and residency requirement as
 * moe_decode_layer; shapes outside the one-shot plan return
 * MOE_ERR_UNSUPPORTED.  1 <= layers <= 4096. */
int moe_decode_stack(const uint16_t* x0, int T, double eps, int layers, const uint16_t* wr_bf16,
                     const float* bias, int E, int k, const void* const* expert_ptrs, moe_expert_shape s,
                     int32_t* idx, float* weights, float* logits, uint16_t* x_out, float* y,
                     void* workspace, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Decode without allocation.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory on the decode
 * path, such as a plugin that a host framework hands only its input and
 * output buffers, or a serving loop that must never enter an allocator.  It
 * computes exactly what moe_experts_decode computes, with the same arguments
 * minus the workspace: the scratch is a static device array inside the
 * library of moe_experts_decode_noalloc_limit() bytes (2 MiB), held by every
 * GPU that loads the library until the process exits.
 *  - A call whose moe_experts_decode_workspace(T, k, s) exceeds that limit
 *    returns MOE_ERR_WORKSPACE_TOO_SMALL and launches nothing.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call shares the one array per device: calls whose kernels overlap
 *    on the GPU (other streams, other threads) race and give wrong results.
 *    The part that must start at zero is cleared by each call on `stream`,
 *    after every argument check has passed (a rejected call leaves the array
 *    as it was and returns what moe_experts_decode would).
 *  - The residency requirement of moe_experts_decode applies.
 *  - No cudaMalloc, cudaFree or other allocating routine is called. */
size_t moe_experts_decode_noalloc_limit(void);
int moe_experts_decode_noalloc(const uint16_t* x_bf16, const int32_t* idx, const float* weights,
                               int T, int k, const void* const* expert_ptrs, int E,
                               moe_expert_shape s, float* y, int32_t* dev_status, void* stream);

/* Bucketing of routed pairs by expert (first page, "The engine", item 5:
 * the whole prompt runs through a layer at once; second page, "v3": each
 * expert's tokens are found by comparing the index tensor with the expert).
 * idx [T x k] int32 input.  counts [E], offsets [E+1] (exclusive scan of
 * counts), pairs [T*k]: the pair ids p = t*k + j grouped by expert, ascending
 * p inside each group.  Bit-reproducible.  An index outside [0, E) sets
 * MOE_DEV_BAD_INDEX in dev_status (if given) and the pair is dropped.
 * workspace: at least moe_bucket_workspace(T, k, E) bytes. */
size_t moe_bucket_workspace(int T, int k, int E);
int moe_bucket_by_expert(const int32_t* idx, int T, int k, int E, int32_t* counts,
                         int32_t* offsets, int32_t* pairs, void* workspace,
                         size_t ws_bytes, int32_t* dev_status, void* stream);

/* Workspace bytes moe_experts_grouped needs. */
size_t moe_experts_grouped_workspace(int T, int k, int E, moe_expert_shape s);

/* Prompt path: the same layer for many tokens as a grouped contraction on
 * the tensor cores (tcgen05, FP32 accumulation in TMEM).  Gate/up operands
 * are FP16 for NVFP4 records (weights exact; x converted from BF16, exact for
 * magnitudes in [2^-14, 65504], below that rounded to an FP16 subnormal, at
 * or above 65520 flagged with MOE_DEV_FP16_RANGE) and BF16 for MXFP4; the
 * down projection is BF16.
 * Same arguments and output as moe_experts_decode, except:
 *  - the SwiGLU intermediate silu(g) * u is rounded to BF16 before the down
 *    projection (it is a BF16 MMA operand);
 *  - the k contributions to y[t] are accumulated with FP32 atomic adds, so
 *    the order of the additions (and the last bits of y) may vary between
 *    runs.
 * Only MOE_FMT_NVFP4 and MOE_FMT_MXFP4 records with H % 128 == 0 and
 * I % 128 == 0 are accepted. */
int moe_experts_grouped(const uint16_t* x_bf16, const int32_t* idx, const float* weights,
                        int T, int k, const void* const* expert_ptrs, int E,
                        moe_expert_shape s, float* y, void* workspace, size_t ws_bytes,
                        int32_t* dev_status, void* stream);

/* FP8 row-scaled matrix-vector (first page, "Why this model": large matrices
 * stored in FP8 with one scale per row; "The engine", item 4: their own GEMV
 * kernel).  w_e4m3 [M x K] E4M3FN bytes, row_scale [M] FP32, x_bf16 [K];
 * y[m] = row_scale[m] * sum_k e4m3(w[m,k]) * x[k], FP32 accumulation.
 * K % 16 == 0; w and x 16-B aligned.
 * For K <= 4096 the launch is a programmatic dependent launch that reads w
 * before it waits for the previous kernel of the stream (x and row_scale only
 * after): w is a weight that no kernel of the stream writes in the call's
 * immediate past, as for model parameters; a caller that has just produced w
 * on the same stream synchronises (or records an event) first. */
int fp8_rowscale_gemv(const uint8_t* w_e4m3, const float* row_scale, const uint16_t* x_bf16,
                      int M, int K, float* y, void* stream);

/* Static text for a moe_status value. */
const char* moe_status_string(int status);

/* Test hook for the bounded waits of moe_decode_layer and of
 * moe_experts_decode's one-shot kernel, so that a test can make a wait run
 * out without faulting or hanging the GPU.  The pages have no counterpart.
 * wait_ns: the limit of every bounded wait in those kernels (0 restores the
 *   default of 2 s; otherwise 1 us .. 10 s).
 * barrier_extra_arrivals: 0, or 1 to make every grid barrier wait for one
 *   arrival more than the grid makes -- it then runs out after wait_ns, the
 *   launch sets MOE_DEV_TIMEOUT and writes NaN outputs.  Zero the workspace
 *   again before the next call.
 * The setting is process-wide and applies to launches made after the call.
 * Returns MOE_ERR_INVALID_ARG for values outside those ranges. */
int moe_test_set_wait_limit(unsigned long long wait_ns, int barrier_extra_arrivals);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
