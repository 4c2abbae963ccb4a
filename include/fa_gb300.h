/*
 * fa_gb300.h — C ABI of the GB300 (sm_103a) fused exact attention: the
 * forward (bf16, and on FP8 operands), its backward, and the FP8 quantiser.
 *
 * The operation.  For every batch b, head h and query row i,
 *
 *     O[b,h,i,:] = sum_j softmax_j( scale * Q[b,h,i,:] . K[b,h,j,:] ) * V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp( scale * Q[b,h,i,:] . K[b,h,j,:] )
 *
 * where j runs over 0..N-1, or over 0..i when causal (top-left mask, key j
 * visible to query i iff j <= i).  This is Eq. 4.1 of "4 Triton and Custom
 * Kernels" (aisyseng.dev, section 4.7), with the logsumexp output of
 * "FlashAttention 2 from PyTorch to Triton" (section "What I am building")
 * and "FlashAttention and kernels." (section "FlashAttention's forward pass").
 * The kernel computes it tile by tile with the online softmax (running row
 * maximum, running row sum, rescaled fp32 accumulator, exp2), so the N x N
 * score matrix never reaches device memory.  fa_bwd computes the gradients
 * of O with respect to Q, K and V by the same tiles, rebuilding P from LSE.
 *
 * Conventions shared by every entry point:
 *   - Pointers named q, k, v, o, lse are DEVICE pointers on the current device.
 *     The caller owns every buffer it passes.  The library's own device
 *     memory is a status word per device (static) and, per stream, one
 *     workspace of 2 x (SMs, at most 256) x 256 x 129 fp32 values (about
 *     40 MB on a GB300) plus 2048 counters for the parts of split work
 *     items, allocated (and its counters zeroed) on the
 *     first fa_fwd on that stream that splits an item (or splits the keys
 *     of a decode call, whose chunk partials use its first part), with the
 *     counters cleared on that stream, and kept until fa_release_stream or
 *     the end of the process; and, per stream, the backward's workspace (see
 *     fa_bwd).  fa_fwd_noalloc and fa_quantize_fp8 allocate nothing.  Calls
 *     on one stream reuse its workspaces in stream order; calls on different
 *     streams never share one.  A caller that creates many short-lived
 *     streams releases each one's workspaces with fa_release_stream.
 *   - The library keeps per-device state for the life of the process (the
 *     device's properties, the status word's and fa_fwd_noalloc's scratch
 *     addresses, the workspaces).  It does not survive cudaDeviceReset: do
 *     not call the library on a device after resetting it.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream) and return a status code.
 *   - Status 0 is FA_OK.  A negative status is returned for an error found
 *     before launch; nothing is launched and the outputs are left untouched.
 *     No entry point aborts, throws or prints.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1,    /* B, H or N < 1; d not 64 or 128; causal not 0/1;
                                 scale not finite or <= 0; sizes overflowing indices */
  FA_ERR_NULL = -2,           /* a required pointer is NULL */
  FA_ERR_ALIGN = -3,          /* q, k, v or o not 16-byte aligned, or lse not 4-byte aligned */
  FA_ERR_ALIAS = -4,          /* o or lse overlaps an input, or o overlaps lse */
  FA_ERR_DEVICE = -5,         /* current device is not compute capability 10.3 (sm_103a) */
  FA_ERR_LAUNCH = -6,         /* a CUDA call failed (tensor-map encoding, attribute, launch) */
  FA_ERR_DEVICE_TIMEOUT = -7, /* a pipeline wait inside the kernel gave up (see fa_get_device_status) */
  FA_ERR_SCRATCH = -8         /* fa_fwd_noalloc: the device's work plan needs more than its static scratch */
};

/*
 * fa_fwd — fused attention forward.
 *
 *   q, k, v : bf16 [B][H][N][d], contiguous (d fastest), read only.
 *   o       : bf16 [B][H][N][d], contiguous; written.  Must not overlap q, k, v or lse.
 *   lse     : fp32 [B][H][N]; written with the natural-log logsumexp of each
 *             row of scaled (and masked) scores.
 *   B, H, N : batch, heads, sequence length (queries = keys = N), each >= 1,
 *             with B*H*N*d < 2^31.
 *   d       : head dimension, 64 or 128.
 *   causal  : 0 = every key visible; 1 = key j visible to query i iff j <= i.
 *   scale   : multiplies Q.K before the softmax (typically 1/sqrt(d)); finite, > 0.
 *   stream  : cudaStream_t as void*.
 *
 * Work division.  A work item is 256 query rows of one (b, h); its cost is
 * the key tiles of 128 its longer half visits.  When every (b, h) has at
 * most 128 query rows, B*H is even and B*H / 2 is at least the number of
 * SMs, an item instead pairs the query rows of two heads (each half of the
 * item streaming its own head's K and V), so that both halves have work.  With more items than SMs
 * (or fewer, but with at least 16 key tiles per SM to share out),
 * the concatenated steps of all items are cut into one equal contiguous
 * range per CTA (at most one CTA per SM); an item cut between two CTAs is computed in parts, each
 * writing O normalised over its own keys and its logsumexp to the stream's
 * workspace; the CTA whose arrival completes an item's parts merges them
 * (O = sum_r exp(L_r - L) O_r, L = ln sum_r exp(L_r)) after its own work, so
 * such a call is one launch.  Otherwise one CTA takes each item.  Without
 * the mask and with N <= 4, the call takes the decode kernels instead (see
 * fa_fwd_rect).  fa_fwd_plan reports the choice.
 *
 * P (the softmax numerators) is rounded to bf16 before the P.V product and O
 * is rounded once to bf16 (round to nearest even) after the fp32 division by
 * the row sum ("How to profile and optimise kernels", the cast of P to bf16).
 * Returns FA_OK or a negative fa_status.  Rows i >= N are never written.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, int causal, float scale, void* stream);

/*
 * fa_fwd_rect — fa_fwd with Nq query rows and Nk keys per (b, h), which may
 * differ.
 *
 *   q, o    : bf16 [B][H][Nq][d], contiguous.
 *   k, v    : bf16 [B][H][Nk][d], contiguous.
 *   lse     : fp32 [B][H][Nq].
 *   causal  : 1 = key j visible to query i iff j <= i (top-left, the
 *             convention non-square causal attention is checked against in
 *             "How to profile and optimise kernels", Round 4); every row
 *             sees key 0, so no row is ever fully masked.
 * Few query rows over many keys (the decode shape) is the case this opens.
 *   - causal = 0 and Nq <= 4 (and B*H <= 65535): the decode kernels, on the
 *     CUDA cores, since the work is bound by reading K and V once.  The keys
 *     of each (b, h) are cut into equal chunks (about eight CTAs per SM in
 *     all, each chunk a multiple of 64 keys), each CTA streams its chunk
 *     through shared memory and writes O normalised over the chunk and its
 *     logsumexp to the stream's workspace, and the CTA whose arrival
 *     completes a (b, h) (one counter per (b, h) among the workspace's
 *     counters) merges its chunks in the same launch (O = sum_c exp(L_c - L)
 *     O_c, L = ln sum_c exp(L_c)); with B*H above the 2048 counters a second
 *     launch merges instead.  One chunk: written directly.  P stays in fp32
 *     here: nothing is rounded before P.V.
 *   - otherwise the attention kernel of fa_fwd: when there are no more work
 *     items than SMs, the keys of each item are split over several CTAs (at
 *     least 16 key tiles each) and the parts merged in the same launch.
 * Errors as fa_fwd, with Nq and Nk each >= 1 and B*H*Nq*d, B*H*Nk*d < 2^31.
 */
int fa_fwd_rect(const void* q, const void* k, const void* v, void* o, float* lse,
                int B, int H, int Nq, int Nk, int d, int causal, float scale, void* stream);

/*
 * fa_fwd_noalloc — fa_fwd (same arguments, kernels, work division and
 * results, bit for bit) with no device allocation at any call: the parts of
 * split items go to one static scratch array of FA_NOALLOC_SCRATCH_BYTES per
 * device instead of the per-stream workspace.  One exception: the decode
 * shapes (causal = 0 and N <= 4), which fa_fwd sends to the decode kernels,
 * run the attention kernel here (its results then agree with fa_fwd's within
 * the bf16 path's tolerance, not bit for bit).  The paper has no counterpart; it is
 * for callers that must not allocate during a call, such as a server that
 * reserves its whole memory budget at start-up, or one that cannot afford a
 * cudaMalloc/cudaFree blocking on work queued on other streams.
 *
 *   - Limit: the scratch holds the workspace of up to FA_NOALLOC_MAX_CTAS
 *     CTAs (two parts of 256 rows x 129 fp32 each per CTA, and eight arrival
 *     counters per split item); the work plan
 *     uses one CTA per SM.  On a device with more SMs than that, a call
 *     that splits items returns FA_ERR_SCRATCH and launches nothing.
 *     Problem sizes are limited as for fa_fwd.
 *   - The arrival counters must start at zero: the first call's set-up
 *     clears the scratch, and every call leaves the counters at zero again.
 *     A call whose kernel gave up on a wait (FA_ERR_DEVICE_TIMEOUT) may
 *     leave them non-zero; fa_get_device_status, which reports that, clears
 *     them.  Nothing else has to start at any value.
 *   - The scratch is shared by every call on the device: calls whose work
 *     overlaps on the GPU (e.g. on two streams at once) race on it and give
 *     wrong results.  Calls on one stream are ordered and safe.
 *   - The first call on a device does that device's set-up (device query,
 *     the kernels' shared-memory attribute, the scratch's address); make
 *     that first call before any stream capture.  The array lives in a
 *     module of its own, loaded (and its device memory reserved by the CUDA
 *     runtime) when the first call looks up its address, or when the
 *     context is created if modules load eagerly.
 * Returns FA_OK or a negative fa_status (the errors of fa_fwd, plus
 * FA_ERR_SCRATCH).
 */
#define FA_NOALLOC_MAX_CTAS 160
#define FA_NOALLOC_SCRATCH_BYTES ((160u * 2u * 256u * 129u + 2048u) * 4u) /* 42,278,912 bytes */
int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, int causal, float scale, void* stream);

/*
 * fa_fwd_plan — the work division fa_fwd_rect (fa_fwd: Nq = Nk = N) would use
 * on the current device for these sizes (no pointer is needed and nothing
 * is launched or allocated):
 * *num_ctas = the attention kernel's grid, *num_split_items = items computed
 * in parts (merged inside the same launch).  For the decode kernels' shapes:
 * *num_ctas = chunks x B x H, *num_split_items = B x H when the keys are cut
 * into more than one chunk, else 0.  The paper has no counterpart;
 * it exists so that callers can see how the work is divided.  Returns FA_OK, FA_ERR_NULL (an output pointer is NULL),
 * FA_ERR_INVALID_ARG (sizes as for fa_fwd), FA_ERR_DEVICE or FA_ERR_LAUNCH.
 */
int fa_fwd_plan(int B, int H, int Nq, int Nk, int d, int causal, int* num_ctas,
                int* num_split_items);

/* Human-readable name of a status code; never NULL, static storage. */
/*
 * fa_bwd — attention backward: the gradients of O = softmax(scale Q K^T [mask]) V
 * with respect to Q, K and V, for an upstream gradient dO.
 *
 *   q, o, dout : bf16 [B][H][Nq][d], contiguous, read only (o is the forward's output).
 *   k, v       : bf16 [B][H][Nk][d], contiguous, read only.
 *   lse        : fp32 [B][H][Nq], the forward's natural-log logsumexp, read only.
 *   dq         : bf16 [B][H][Nq][d]; written.
 *   dk, dv     : bf16 [B][H][Nk][d]; written.  No output may overlap an input or another output.
 *   B, H, Nq, Nk, d, causal, scale : as for fa_fwd_rect (the same values the
 *             forward used; causal is the top-left mask), with
 *             B*H*ceil(Nq/64)*64*d < 2^31, B*H*Nk*d < 2^31, B*H <= 65535 and,
 *             with causal = 1, ceil(Nk/128) <= 65535.
 *   stream     : cudaStream_t as void*.
 *
 * The method is the recompute-from-L backward of "FlashAttention and
 * kernels." (gtadkapally.com, section "The backward pass: recompute instead
 * of remember"): P = exp(scale Q K^T - L) rebuilt tile by tile, never stored;
 * D = rowsum(dO * O) once per query row; dV = P^T dO, dP = dO V^T,
 * dS = P * (dP - D), dQ = scale dS K, dK = scale dS^T Q.  P and dS are rounded
 * to bf16 before their products; every product accumulates in fp32; the
 * outputs are rounded once to bf16.  dQ sums the contributions of all key
 * blocks in an fp32 accumulator (reductions performed in L2) in the order
 * they arrive, so its last bit may differ between runs; dK and dV are
 * deterministic.
 *
 * Three launches on `stream`: prep (D, L in log2 units, accumulator zeroed),
 * the backward kernel (one CTA per (b, h, 128-key block)), and the dQ
 * conversion.  Device memory: besides the status word, one workspace per
 * stream of B*H*Nq*d*4 + 2*B*H*ceil(Nq/64)*64*4 bytes (rounded up to 256),
 * allocated on the first call on that stream and grown (after synchronising
 * the stream) when a call needs more; kept until the process exits.
 *
 * Returns FA_OK or a negative fa_status: FA_ERR_INVALID_ARG, FA_ERR_NULL,
 * FA_ERR_ALIGN (a bf16 tensor not 16-byte aligned, lse not 4-byte aligned),
 * FA_ERR_ALIAS, FA_ERR_DEVICE or FA_ERR_LAUNCH (also when the workspace
 * cannot be allocated).  A kernel wait that gives up is reported by
 * fa_get_device_status, as for the forward.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dout, void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d,
           int causal, float scale, void* stream);

/*
 * fa_quantize_fp8 — bf16 to FP8 (e4m3) codes with per-block fp32 scales, in
 * the layouts fa_fwd_fp8 reads.  A block of rows shares one scale
 * s = amax / 448 (s = 1 for an all-zero block); each element becomes the
 * e4m3 value nearest to x / s (ties to even, saturating at +-448; the
 * division in fp32).  The pages name FP8 with per-block scaling
 * ("FlashAttention and kernels.", section "FlashAttention-2, -3, and what
 * came after") without fixing the blocks; the reading here:
 *
 *   mode 0 (Q, K): x bf16 [B][H][N][d] -> x8 [B][H][N][d] (one byte each),
 *                  scales [B][H][ceil(N/128)], one per 128 rows;
 *   mode 1 (V):    x bf16 [B][H][N][d] -> x8 [B][H][d][N_pad], transposed,
 *                  N_pad = ceil(N/128)*128, keys past N zero;
 *                  scales [B][H], one per head (V's scale has to factor out
 *                  of the sum over key tiles).
 *
 *   d: 64 or 128.  x, x8 16-byte aligned, scales 4-byte aligned, device
 *   pointers, no overlaps.  Four launches on `stream` (the scales are
 *   zeroed, then amax, codes, scales).  Returns FA_OK or a negative fa_status.
 */
int fa_quantize_fp8(const void* x, void* x8, float* scales, int B, int H, int N, int d, int mode,
                    void* stream);

/*
 * fa_fwd_fp8 — the forward on FP8 operands: O and LSE (as fa_fwd) of
 * attention on the dequantised inputs q8 * sQ, k8 * sK, v8 * sV, from the
 * layouts fa_quantize_fp8 writes (q8, k8 mode 0; vt8 mode 1).  d = 128.
 * S = Q K^T and O += P V run on the tensor core's e4m3 instruction
 * (kind::f8f6f4) with fp32 accumulation; P is rounded to e4m3 before P V
 * (P <= 2^8 by the forward's lazy maximum, inside e4m3's range); the scales
 * enter the exponent (sQ sK) and the final division (sV).  Same work
 * division, workspace and errors as fa_fwd; o bf16 [B][H][N][128] and lse
 * fp32 [B][H][N] must not overlap an input.
 */
int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale,
               const float* k_scale, const float* v_scale, void* o, float* lse, int B, int H, int N,
               int d, int causal, float scale, void* stream);

const char* fa_strerror(int code);

/*
 * fa_get_device_status — reports whether any kernel launched by this library
 * on the current device gave up on a pipeline wait (every wait inside the
 * kernel is bounded in time; on expiry the kernel records the failure, stops
 * its pipeline, releases tensor memory and exits instead of hanging).
 * Reads the device's status word on `stream` (after the work queued there)
 * and returns FA_OK or FA_ERR_DEVICE_TIMEOUT.  On a timeout it then waits for
 * the whole device (cudaDeviceSynchronize), and clears the status word and
 * the split-item counters of every workspace and of fa_fwd_noalloc's scratch
 * on `stream`, waiting for the clears; call it then with no other call of
 * this library in flight on the device (it is the recovery path).  Returns
 * FA_ERR_LAUNCH if a CUDA call fails.
 */
int fa_get_device_status(void* stream);

/*
 * fa_release_stream — frees the workspaces (forward and backward) that this
 * library keeps for `stream` on the current device, after synchronising the
 * stream.  A later call on the stream allocates them again.  Call it before
 * destroying a stream the library has used, when streams are short-lived.
 * The paper has no counterpart.  Returns FA_OK, or FA_ERR_LAUNCH if a CUDA
 * call fails.
 */
int fa_release_stream(void* stream);

/*
 * fa_watchdog_selftest — launches one small forward whose load warp is told
 * never to deliver its K/V tiles, with every wait limited to `limit_ms`
 * milliseconds, so that the bounded waits run out on purpose.  q, k, v, o
 * and lse are as for fa_fwd with B=H=1, N=128, d=64 (caller-owned, device).
 * Synchronises `stream` and returns what fa_get_device_status then reports
 * (FA_ERR_DEVICE_TIMEOUT when the watchdog works), or a launch error.
 * Test hook for the failure-detection path; never used by fa_fwd.
 */
int fa_watchdog_selftest(const void* q, const void* k, const void* v, void* o, float* lse,
                         int limit_ms, void* stream);

/* Library version as 10000*major + 100*minor + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
