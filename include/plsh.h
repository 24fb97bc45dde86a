/*
 * plsh.h -- C ABI of the Positional LSH approximate-ALiBi attention library
 * for GB300 (sm_103a).
 *
 * The method ("Positional LSH: Binary Block Matrix Approximation for
 * Attention with Linear Biases", Wolfson & Wagner; technical summary):
 *   Methodology 1   L*_ij = exp(-|i-j|/sigma) is a Laplacian kernel on token
 *                   positions.  A random-binning hash of the integer positions
 *                   splits 0..n-1 into contiguous bins; M(h) is 1 where i and
 *                   j share a bin, and L* = E_h[M(h)].
 *   Methodology 2   (Theorem 2.1) the mean M~ of s i.i.d. masks approximates
 *                   L*; bin widths follow a Gamma law.
 *   Methodology 3   (Theorem 2.2) ALiBi attention becomes s sets of short
 *                   block attentions with no positional bias:
 *                     T~ = D~^-1 (M~ o exp(QK^T/sqrt(d))) V,
 *                   numerator and row sums both averaged over the s masks.
 *
 * Conventions shared by every call:
 *   - Tensors are [B, H, n, d] contiguous row-major, on the CUDA device
 *     that is current when the call is made, 16-byte aligned.  Query head h
 *     reads KV head h / (Hq / Hkv) (contiguous GQA groups).
 *   - The caller owns Q, K, V and O.  The library owns plsh_bins handles and
 *     its per-device work-queue state.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     is asynchronous on it except where a comment says it synchronises.
 *   - Arguments are validated before anything is launched; on a validation
 *     error nothing is written and the status says why (plsh_last_error()
 *     holds a message for the calling thread).  No call aborts or prints.
 */
#ifndef PLSH_H_
#define PLSH_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PLSH_OK = 0,
  PLSH_ERR_INVALID = 1,      /* bad argument: shape, dtype, range, pointer  */
  PLSH_ERR_CUDA = 2,         /* a CUDA runtime/driver call failed           */
  PLSH_ERR_NOMEM = 3,        /* device or host allocation failed            */
  PLSH_ERR_TIMEOUT = 4,      /* a device-side bounded wait ran out          */
  PLSH_ERR_UNSUPPORTED = 5,  /* valid request the library does not serve    */
  PLSH_ERR_RANGE = 6         /* an input value beyond the range the kernel
                                computes in (V beyond +-65504 on the
                                tensor-core path), found on the device      */
} plsh_status;

/* Which kernel serves an attention call (plsh_attn_path). */
typedef enum { PLSH_PATH_CUDA_CORES = 0, PLSH_PATH_TENSOR_CORES = 1 } plsh_path;

typedef enum { PLSH_F32 = 0, PLSH_BF16 = 1 } plsh_dtype;

/* A device tensor [B, H, n, d], contiguous, element type `dtype`.
 * `data` is a device pointer the caller owns. */
typedef struct {
  void* data;
  int32_t dtype;   /* plsh_dtype */
  int64_t B, H, n, d;
} plsh_tensor;

/* Opaque set of s bin partitions per head (one per hash), resident on one
 * device.  Owns its device memory; reusable by any number of attention
 * calls (the same draws serve every batch element and layer). */
typedef struct plsh_bins plsh_bins;

/*
 * plsh_sample_bins -- draw s random-binning hashes per head and build their
 * bins on the device (Methodology 1-2).
 *
 * For head h and sample t the counter-based generator Philox4x32-10 (key =
 * seed, counter = (t, h, 0, 0)) gives U0, U1, U2 = (x + 0.5) 2^-32; the width
 * is w = sigma_h (-ln U0 - ln U1) ~ Gamma(shape 2, scale sigma_h) and the
 * offset u = w U2 ~ U(0, w).  Bin starts are 0 and ceil(u + k w) for
 * k = 0, 1, ... below n, u + k w one fused multiply-add (every position its
 * own bin when w < 1).  The arithmetic is fp64, each operation (a fused
 * multiply-add counts as one) rounded once, so the starts agree bit for bit
 * with any other implementation of the same recipe.
 *
 *   n        sequence length, 1 <= n < 2^31
 *   sigma_h  host array [H], each finite and > 0 (sigma = 1 / ALiBi slope)
 *   H        number of query heads, >= 1
 *   s        hashes per head, 1 <= s <= 64
 *   seed     64-bit generator key
 *   out      receives a new handle (free with plsh_bins_free)
 * Allocates device memory (synchronous allocation), then launches the
 * sampler on `stream`.  On error *out is left unchanged.
 */
plsh_status plsh_sample_bins(int64_t n, const double* sigma_h, int32_t H,
                             int32_t s, uint64_t seed, void* stream,
                             plsh_bins** out);

/*
 * plsh_bins_resample -- redraw an existing handle in place with new sigma_h
 * and seed (same n, H, s).  Allocates nothing; fully asynchronous.  The
 * previous contents must no longer be in use by work queued on other
 * streams.
 */
plsh_status plsh_bins_resample(plsh_bins* bins, const double* sigma_h,
                               uint64_t seed, void* stream);

/*
 * plsh_bins_from_host -- build a handle from explicit bin boundaries (for
 * deterministic variants such as fixed blocks, or draws made elsewhere).
 *   offsets  host int64 [H*s + 1]; hash (h, t) owns
 *            starts[offsets[h*s+t] .. offsets[h*s+t+1])
 *   starts   host int32; each hash's list begins with 0, strictly increases
 *            and ends with the terminal n
 * Validated on the host; synchronous upload.
 */
plsh_status plsh_bins_from_host(int64_t n, int32_t H, int32_t s,
                                const int64_t* offsets, const int32_t* starts,
                                void* stream, plsh_bins** out);

/*
 * plsh_bins_fixed -- deterministic fixed blocks in place of random hashes (the
 * "fixed blocks" baseline of the summary's Mistral fine-tuning experiment,
 * Experimental validation): hash t of head h cuts 0..n-1 into contiguous
 * blocks of width_h[h] positions, shifted by o = floor(t * width_h[h] / s),
 * i.e. bin starts {0} u {o + k * width_h[h] : k >= 0} inside [1, n).  With
 * s = 1 these are plain blocks [0, w), [w, 2w), ...; larger s averages s
 * evenly shifted grids, the deterministic counterpart of the random offsets.
 *   width_h: host array [H], every entry >= 1.  1 <= s <= 64, 1 <= n < 2^31.
 * The records are built on the device in closed form; the call waits for it
 * (the host arrays it uploads are its own).  The handle is used exactly like
 * one from plsh_sample_bins (plsh_bins_draws reports w = width, u = o);
 * plsh_bins_resample on it draws random bins.
 */
plsh_status plsh_bins_fixed(int64_t n, const int32_t* width_h, int32_t H, int32_t s,
                            void* stream, plsh_bins** out);

/*
 * plsh_alibi_attn_backward -- gradients of sum(T~ * dO) with respect to Q, K
 * and V (the backward pass of plsh_alibi_attn, Methodology 3's estimator with
 * the multiplicities c_ij held fixed):
 *   P_ij = c_ij e^{S_ij} / sum_j c_ij e^{S_ij},  dP_ij = dO_i . v_j,
 *   dS_ij = P_ij (dP_ij - sum_l P_il dP_il),
 *   dQ_i = sum_j dS_ij k_j / sqrt(d),  dK_j = sum_i dS_ij q_i / sqrt(d),
 *   dV_j = sum_i P_ij dO_i,
 * a KV head collecting the sums of every query head that reads it.
 *   Q, dO, dQ [B,Hq,n,d]; K, V, dK, dV [B,Hkv,n,d]; one dtype (PLSH_BF16 or
 *   PLSH_F32), d in {64, 128}; bins and causal as for plsh_alibi_attn.
 * Tensor cores (bf16, d = 128, s <= 16, Hq / Hkv <= 64; plsh_attn_path names
 * the path): the forward kernel in a row statistics mode writes each row's
 * max, sum and Delta_i = dO_i . O_i, then a kernel per (batch, KV head, key
 * tile) forms S^T, dP^T, dV, dK and dS K with tcgen05 products (P and dS
 * rounded to bf16, fp32 accumulation), the dS K rows added to an fp32 dQ
 * accumulator by TMA reductions and converted to bf16 at the end.
 * CUDA cores (every other case), fp32 accumulation, no atomics: a warp per
 * row computes the row's max, sum and sum_j P_ij dP_ij and dQ_i; a warp per
 * key then sums dK_j and dV_j over the rows whose bins contain it.
 * Scratch (2 or 3 B Hq n floats of row statistics, plus B Hq n d floats of
 * dQ accumulator on the tensor cores) lives in a device buffer the library
 * keeps per device between calls, grown on demand in stream order on
 * `stream` (from the device's stream-ordered memory pool); calls on
 * different streams are ordered on it by an event.
 * Asynchronous on `stream`.
 */
plsh_status plsh_alibi_attn_backward(const plsh_tensor* Q, const plsh_tensor* K,
                                     const plsh_tensor* V, const plsh_tensor* dO,
                                     const plsh_bins* bins, int32_t causal, plsh_tensor* dQ,
                                     plsh_tensor* dK, plsh_tensor* dV, void* stream);

/*
 * plsh_alibi_attn_backward_lse -- the same gradients from the forward pass's
 * output O and log-sum-exp lse (written by plsh_alibi_attn_lse for the same
 * Q, K, V, bins and causal), as a training step has them: the rows'
 * Delta_i = dO_i . O_i comes from O (bf16, as stored) in a pass over the rows
 * instead of a recomputation of the forward pass.
 *   O [B,Hq,n,d] with Q's shape and dtype; lse [B*Hq*n] fp32 device memory.
 * Tensor cores only (bf16, d = 128, s <= 16, Hq / Hkv <= 64): other inputs
 * return PLSH_ERR_UNSUPPORTED.  Scratch, ordering and errors as for
 * plsh_alibi_attn_backward.  Asynchronous on `stream`.
 */
plsh_status plsh_alibi_attn_backward_lse(const plsh_tensor* Q, const plsh_tensor* K,
                                         const plsh_tensor* V, const plsh_tensor* O,
                                         const float* lse, const plsh_tensor* dO,
                                         const plsh_bins* bins, int32_t causal, plsh_tensor* dQ,
                                         plsh_tensor* dK, plsh_tensor* dV, void* stream);

/*
 * plsh_bias_error -- the bias of the averaged mask for head h of `bins`:
 * ||L* - M~||_max and ||L* - M~||_2 with L*_ij = e^{-|i-j|/sigma} (Problem
 * statement) and M~ = (1/s) sum_t M(h_t) (Methodology 1-2), the two norms the
 * summary's convergence experiment follows against s (Results).  Neither
 * n x n matrix is formed: the max norm is exact (per row over its key
 * envelope); the spectral norm, the largest eigenvalue magnitude of the
 * symmetric difference, is estimated by `lanczos_iters` Lanczos steps from a
 * start vector drawn from `seed`, with O(n s) products (the Laplace kernel as
 * two linear recurrences, the mask through prefix sums).  fp64 throughout.
 *   sigma > 0 (the scale L* is taken at), 0 <= h < H,
 *   2 <= lanczos_iters <= 1000 when spectral is requested.
 *   max_abs, spectral: host outputs; either may be NULL to skip it.
 * Blocks until done (device scratch of 6 n doubles, allocated per call).
 */
plsh_status plsh_bias_error(const plsh_bins* bins, double sigma, int32_t h,
                            int32_t lanczos_iters, uint64_t seed, double* max_abs,
                            double* spectral, void* stream);

/*
 * plsh_bins_share_groups -- hashes shared across a GQA group: bins for Hq
 * query heads in which head h uses every hash (records, draws and scale) of
 * head floor(h / (Hq / G)) of `src`, G = src's number of heads, Hq % G == 0.
 * Drawn with one scale per KV group (plsh_sample_bins with G heads), the heads
 * of a group then cut the positions identically, so the key envelopes of two
 * heads of one group coincide.  A variant outside the summary's method (each
 * of its heads draws its own hashes).  Device-to-device copies; the call
 * waits for them.  plsh_bins_resample on the result draws per-head hashes.
 */
plsh_status plsh_bins_share_groups(const plsh_bins* src, int32_t Hq, void* stream,
                                   plsh_bins** out);

/* Shape of a handle.  n_entries (bins + terminals over all hashes) needs the
 * device contents: this call synchronises `stream` when n_entries != NULL. */
plsh_status plsh_bins_info(const plsh_bins* bins, int64_t* n, int32_t* H,
                           int32_t* s, int64_t* n_entries, void* stream);

/*
 * plsh_bins_to_host -- copy the bin boundaries back in the plsh_bins_from_host
 * layout.  offsets [H*s+1]; starts must hold `cap` entries (query the size
 * with plsh_bins_info).  Synchronises `stream`.
 */
plsh_status plsh_bins_to_host(const plsh_bins* bins, int64_t* offsets,
                              int32_t* starts, int64_t cap, void* stream);

/* Draws (w, u) of every (h, t), host arrays [H*s] (either may be NULL).
 * Synchronises `stream`. */
plsh_status plsh_bins_draws(const plsh_bins* bins, double* w, double* u,
                            void* stream);

/* Frees the handle's device memory (synchronises the device first). */
void plsh_bins_free(plsh_bins* bins);

/*
 * plsh_alibi_attn -- approximate ALiBi attention T~ (Methodology 3).
 *
 * For each batch b, query head h and row i, with J_t(i) the bin of i under
 * hash t of head h (clipped to j <= i when causal):
 *   O_i = sum_t sum_{j in J_t(i)} e^{S_ij} v_j / sum_t sum_{j in J_t(i)} e^{S_ij},
 *   S_ij = q_i . k_j / sqrt(d).
 * Computed as sum_j c_ij e^{S_ij} v_j / sum_j c_ij e^{S_ij}, with c_ij the
 * number of hashes that put i and j in one bin.
 *
 *   Q [B,Hq,n,d]; K, V [B,Hkv,n,d]; O [B,Hq,n,d], all the same dtype,
 *   Hq % Hkv == 0, bins->n == n, bins->H == Hq, d in {64, 128}.
 *   causal   non-zero: keys j <= i only.
 * Kernels (plsh_attn_path tells which one a call takes, without launching):
 *   tensor cores  bf16 with d in {64, 128} and s within the kernel's shared
 *                 memory (s <= 52 causal, s <= 29 without the mask; d = 64
 *                 runs zero-padded to 128 columns in shared memory, at the
 *                 cost of d = 128): QK^T in
 *                 bf16, the weights P and V in f16 for P V (every bf16
 *                 value of V up to 65504 is an f16 value; P keeps 11
 *                 significant bits), fp32 accumulation and softmax.  A value of V beyond +-65504 is reported by
 *                 plsh_stream_status() as PLSH_ERR_RANGE (O is then not
 *                 valid); T~ is linear in V, so V scaled down by a power of
 *                 two gives O scaled down by the same power.
 *   CUDA cores    everything else (fp32, larger s): fp32 throughout.
 * Asynchronous on `stream`.  A device-side wait that runs out (a bug, never
 * expected) is reported by the next plsh_stream_status().  The tensor-core
 * path keeps a work-item table per shape and head order on the device
 * (allocated and uploaded on `stream` at the first call of a shape, in stream
 * order; up to 16 are cached, and the least recently used one that no call
 * holds is freed, in stream order behind the work of the calls that used
 * it, when a seventeenth shape arrives).
 */
plsh_status plsh_alibi_attn(const plsh_tensor* Q, const plsh_tensor* K,
                            const plsh_tensor* V, const plsh_bins* bins,
                            int32_t causal, plsh_tensor* O, void* stream);

/*
 * plsh_alibi_attn_lse -- plsh_alibi_attn that also writes every row's
 * base-2 log-sum-exp of its scaled scores with their multiplicities,
 *   lse_i = log2 sum_j c_ij 2^{x_ij},  x_ij = q_i . k_j log2(e) / sqrt(d)
 * (so that T~_i = sum_j c_ij 2^{x_ij - lse_i} v_j), the statistic the backward
 * pass needs (plsh_alibi_attn_backward_lse).
 *   lse [B*Hq*n] fp32 device memory, row (b, h, i) at (b*Hq + h)*n + i.
 * Tensor-core path only (bf16, d in {64, 128}, s within its budget;
 * plsh_attn_path):
 * other inputs return PLSH_ERR_UNSUPPORTED.  O as for plsh_alibi_attn.
 * Asynchronous on `stream`.
 */
plsh_status plsh_alibi_attn_lse(const plsh_tensor* Q, const plsh_tensor* K,
                                const plsh_tensor* V, const plsh_bins* bins, int32_t causal,
                                plsh_tensor* O, float* lse, void* stream);

/*
 * plsh_alibi_attn_noalloc -- plsh_alibi_attn for callers that may not
 * allocate device memory.  The paper has no counterpart: this is a
 * deployment variant, not part of the method.
 *
 * Some callers cannot let a library call cudaMalloc: a serving process that
 * has reserved all of HBM for its own pools (a late allocation would fail or
 * fragment it), or a latency-bound loop where an allocation's implicit
 * device synchronisation is not acceptable.  This entry point computes the
 * same result as plsh_alibi_attn with the same arguments and rules, but keeps
 * its working memory (the work-item table and the work-queue counters) in a
 * fixed array compiled into the library, about 1 MiB per device, held by
 * every device that loads the library until the process exits.  It calls no
 * allocation routine.
 *
 * Limits: bf16, d = 128, s within the tensor-core kernel's shared-memory
 * budget (s <= 52 causal, s <= 29 without the mask), at most 1023 query
 * heads and 65536 work items (one item per two 128-row query tiles:
 * B * Hq * ceil(n/128) / 2, e.g.
 * n = 131072 with 40 heads uses 20480); larger requests return
 * PLSH_ERR_UNSUPPORTED and launch nothing.
 * The first call on each device resolves the array's device address
 * (cudaGetSymbolAddress) and keeps it for the life of the device's primary
 * context (a process that resets the device must not call this entry point
 * again).
 * Every call on a device shares the one array and each call resets its work
 * counters before use, so calls whose kernels overlap on the GPU (different
 * streams without ordering) race and must not be issued.  A device-side wait
 * that runs out (limit: plsh_set_wait_limit_ns) and a value of V beyond
 * +-65504 are recorded in the array's error word, which persists across calls
 * until plsh_noalloc_status() reads and clears it; plsh_stream_status() does
 * not see them.
 */
plsh_status plsh_alibi_attn_noalloc(const plsh_tensor* Q, const plsh_tensor* K,
                                    const plsh_tensor* V, const plsh_bins* bins,
                                    int32_t causal, plsh_tensor* O, void* stream);

/*
 * plsh_noalloc_status -- the error word of plsh_alibi_attn_noalloc on the
 * current device.  Synchronises `stream`, reads the word from the fixed
 * array (no allocation), clears it, and returns PLSH_ERR_TIMEOUT if a wait
 * ran out, else PLSH_ERR_RANGE if a value of V was beyond +-65504, else
 * PLSH_OK, covering every allocation-free call since the last report.  Call
 * it once the calls it should cover are queued on `stream` (or on streams
 * `stream` waits for).
 */
plsh_status plsh_noalloc_status(void* stream);

/*
 * plsh_alibi_attn_host -- plsh_alibi_attn on tensors in host memory.  The
 * paper has no counterpart: this is a deployment variant, not part of the
 * method.
 *
 * Q, K, V and O follow the plsh_alibi_attn rules except that their `data`
 * are host pointers (page-locked memory lets the copies run asynchronously
 * and overlap; pageable memory works but each copy then blocks the calling
 * thread).  The library stages the tensors through device buffers it keeps
 * per device (grown on demand in stream order, behind the previous call of
 * this entry point; held until the process exits) and splits the query rows
 * into up to four chunks on the tensor-core path: chunk c + 1 is copied in
 * and chunk c - 1 copied out, on two copy streams of its own, while the
 * fused kernel runs on chunk c (with
 * the causal mask only the keys up to a chunk's last row are needed before
 * it starts).  The call returns once everything is queued; O is complete on
 * the host when `stream` reaches the point of the call (synchronise it before
 * reading O).  Calls on one device share the staging buffers: issue them on
 * one stream, or order their streams.
 */
plsh_status plsh_alibi_attn_host(const plsh_tensor* Q, const plsh_tensor* K,
                                 const plsh_tensor* V, const plsh_bins* bins, int32_t causal,
                                 plsh_tensor* O, void* stream);

/*
 * plsh_alibi_exact -- exact ALiBi attention T* (the dense comparator, Problem
 * statement: O(n^2) in the bias matrix):
 *   O_i = sum_j e^{S_ij - |i-j|/sigma_h} v_j / sum_j e^{S_ij - |i-j|/sigma_h}
 * over all j (j <= i when causal).  sigma_h: host array [Hq], finite, > 0.
 * Same tensor rules as plsh_alibi_attn.
 */
plsh_status plsh_alibi_exact(const plsh_tensor* Q, const plsh_tensor* K,
                             const plsh_tensor* V, const double* sigma_h,
                             int32_t causal, plsh_tensor* O, void* stream);

/*
 * plsh_alibi_decode -- one decode step of the approximation: row `pos` of T~
 * (Methodology 3) with the causal mask, for a query given on its own against
 * cached keys and values.  With J_t(pos) = [lo_t(pos), pos], lo_t(pos) the
 * start of the bin of pos under hash t of head h,
 *   o = sum_j c_j e^{S_j} v_j / sum_j c_j e^{S_j},  S_j = q . k_j / sqrt(d),
 *   c_j = #{t : lo_t(pos) <= j},  j in [min_t lo_t(pos), pos]:
 * the work is the row's key envelope, O(s b) keys, not pos.
 *
 *   q [B,Hq,1,d]: the query of position pos; o [B,Hq,1,d]: its output.
 *   K, V [B,Hkv,n,d]: the cache; rows above pos are not read.
 *   All the same dtype (PLSH_BF16 or PLSH_F32), d in {64, 128}, Hq % Hkv == 0,
 *   B * Hq <= 65535, bins->n == n, bins->H == Hq, 0 <= pos < n.
 * A CTA serves the query heads of one KV group (up to 8) over one share of
 * the union of their envelopes; the shares' partial results (max, row sum,
 * unnormalised P V) are merged into o.  The partials live in a device buffer
 * the library keeps per device (B * Hq * S * (d + 2) floats, S <= 64 shares
 * chosen so that about 12 CTAs per SM run, at most the 64-key shares of the
 * envelope the widest bins are expected to reach; grown on demand in stream
 * order on `stream`; calls on different streams are ordered on it by an
 * event).  Up to 32 KV groups are listed widest scale first, and on large
 * grids each group takes the shares its own expected envelope wants.  Both
 * kernels of a call start as programmatic dependents of the kernel before
 * them on `stream` (neither touches global memory before it completes).
 * Asynchronous on `stream`; errors in the arguments return before any launch.
 */
plsh_status plsh_alibi_decode(const plsh_tensor* q, const plsh_tensor* K,
                              const plsh_tensor* V, const plsh_bins* bins, int64_t pos,
                              plsh_tensor* o, void* stream);

/* Synchronises `stream`, then reports CUDA errors and the library's device
 * error flag, clearing the flag: PLSH_ERR_TIMEOUT when a bounded device wait
 * ran out, else PLSH_ERR_RANGE when a tensor-core attention call met a value
 * of V beyond +-65504. */
plsh_status plsh_stream_status(void* stream);

/*
 * plsh_attn_path -- the kernel plsh_alibi_attn (bins != NULL) or
 * plsh_alibi_exact (bins == NULL) takes for a query tensor of Q's shape and
 * dtype, written to *path (a plsh_path).  Launches nothing, allocates
 * nothing; PLSH_ERR_INVALID for a NULL Q or path.
 */
plsh_status plsh_attn_path(const plsh_tensor* Q, const plsh_bins* bins, int32_t causal,
                           int32_t* path);

/* Debug knob: limit in nanoseconds of every device-side wait launched after
 * this call on the current device (0 restores the default of 2 s). */
plsh_status plsh_set_wait_limit_ns(uint64_t ns);

/*
 * plsh_set_split_parts -- how the tensor-core attention calls on the current
 * device cut long work items over their key range (the varlen scheduling
 * step: items are pairs of 128-row query tiles, each item's key envelope is
 * found on the device from its rows' bins).
 *   0   automatic (the default): an item whose expected key tiles exceed
 *       half the call's per-SM share (at least 2) is cut into parts of at
 *       most that size, so that no single item outlasts the others;
 *   1   never cut;
 *   2..16  cut every item into that many parts (a tuning and testing knob).
 * Each part covers a consecutive range of its item's key tiles (a part past
 * the envelope does nothing); parts write their unnormalised P V, running max
 * and row sum to a library-owned workspace and a second kernel combines them
 * into O.  Calls made afterwards use the setting; the workspace is allocated
 * with the item table of a shape.
 */
plsh_status plsh_set_split_parts(int32_t parts);

const char* plsh_status_string(plsh_status status);

/* Message of the last error raised on the calling thread ("" if none). */
const char* plsh_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PLSH_H_ */
