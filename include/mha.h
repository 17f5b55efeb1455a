/*
 * mha.h — C ABI of libmha.so: fused causal multi-head attention forward for
 * NVIDIA GB300 (sm_103a).
 *
 * The operation is the masked multi-head attention of the page "Hand-written
 * masked multi-head attention CUDA kernel: underlying logic and practice"
 * (xdnf.cn/news/357253), section 2:
 *
 *     O = softmax(scale * Q K^T + M) V,   M[i][j] = 0 if j <= i, -inf otherwise
 *
 * (the page prints the last product as "A V^T"; A V is the product whose
 * dimensions agree, and it is what these calls compute).  Section 2.2 of that
 * page fuses the score GEMV, the softmax and the product with V so that
 * scores and probabilities never reach global memory; every call here works
 * that way.  The single-pass running-max/running-sum softmax follows the
 * online-softmax recurrence of the page "Week 4 CUDA notes"
 * (pnsm.cn/news/1831385), section 2.2.
 *
 * Conventions shared by every call:
 *   - Tensors are owned by the caller and live in device memory, contiguous,
 *     with the shapes stated per call.  Every tensor pointer must be 16-byte
 *     aligned (MHA_ERR_MISALIGNED otherwise).
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL means the legacy default stream).  None synchronises the host.
 *   - A call returns MHA_OK or an mha_status.  Argument errors are found on the
 *     host before anything is launched; a launch error is reported as
 *     MHA_ERR_CUDA (the CUDA error is cleared and kept for mha_last_cuda_error).
 *   - Device-side waits inside the kernels are bounded in time; a wait that
 *     runs out sets a device error word instead of hanging, and
 *     mha_get_device_status reports it as MHA_ERR_TIMEOUT.
 *   - LSE, where written, is the natural log of the softmax denominator of
 *     each row: ln(sum over valid keys j of exp(scale * q_i . k_j)), float32.
 */
#ifndef MHA_GB300_H
#define MHA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MHA_OK = 0,
    MHA_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, size overflow   */
    MHA_ERR_UNSUPPORTED = 2,  /* valid but not built: e.g. head dim not 64 or 128 */
    MHA_ERR_MISALIGNED = 3,   /* a tensor pointer is not 16-byte aligned          */
    MHA_ERR_CUDA = 4,         /* a CUDA runtime/driver call or a launch failed    */
    MHA_ERR_TIMEOUT = 5       /* a bounded device wait ran out (see above)        */
} mha_status;

/*
 * Causal (or full) attention prefill, bf16 in and out, fp32 accumulation.
 * Page 3, section 2 (definition) and section 2.2 (fusion and mask j <= i).
 *
 *   Q, K, V : const bf16 [B, H, S, D], contiguous (S query rows = S key rows).
 *   O       : bf16 [B, H, S, D], written.
 *   LSE     : float [B, H, S], written; may be NULL to skip it.
 *   B, H, S : >= 1, with B*H*S*D < 2^31.   D : 64 or 128.
 *   scale   : multiplies Q.K before the mask (1/sqrt(D) for standard attention).
 *   causal  : 1 = key j is used by query i only when j <= i; 0 = every key.
 *   stream  : cudaStream_t.
 *
 * Scores and probabilities stay on chip.  The probabilities are rounded to
 * bf16 before the product with V (the page's section 3.3 stores the operands
 * in 16 bits and accumulates in fp32).  Returns MHA_OK or an mha_status.
 */
int mha_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
            int B, int H, int S, int D, float scale, int causal, void* stream);

/*
 * The same operation on IEEE half precision (f16) inputs and outputs: the
 * page's own kernel is written for half-precision data ("Hand-written masked
 * multi-head attention CUDA kernel", section 3.3).  Arguments and results as
 * mha_fwd, with Q, K, V, O f16 [B, H, S, D].  The probabilities are rounded
 * to f16 before the product with V (both operands of one tensor-core product
 * have the same type); accumulation is fp32.
 */
int mha_fwd_f16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                int B, int H, int S, int D, float scale, int causal, void* stream);

/*
 * mha_fwd with key padding: sequence b of the batch has key_lens[b] valid
 * keys, and key j of sequence b takes part in no row when j >= key_lens[b]
 * (its score is -inf before the softmax, as page "Week 4 CUDA notes" section
 * 2.2 does for padded positions).  With causal = 1 query i uses key j when
 * j <= i and j < key_lens[b].  A row with no valid key (key_lens[b] = 0)
 * gets O = 0 and LSE = -inf.  Key tiles at or past key_lens[b] are neither
 * loaded nor computed.  Query rows i >= key_lens[b] are computed like any
 * other row (they are not masked as queries).
 *
 *   key_lens : const int32 [B] in DEVICE memory; each value in [0, S] (values
 *              outside are clamped to that range on the device).
 *   other arguments as mha_fwd (bf16).
 */
int mha_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                   const int* key_lens, int B, int H, int S, int D, float scale, int causal,
                   void* stream);

/* mha_fwd_varlen on f16 data (the types of mha_fwd_f16). */
int mha_fwd_varlen_f16(const void* Q, const void* K, const void* V, void* O, float* LSE,
                       const int* key_lens, int B, int H, int S, int D, float scale,
                       int causal, void* stream);

/*
 * The same operation with float32 inputs and outputs, computed in fp32 on
 * the CUDA cores (no reduced-precision tensor-core arithmetic anywhere).
 * Page 3 ("Hand-written masked multi-head attention CUDA kernel"), section 2
 * defines the operation and section 3.3 the precision split this path drops:
 * there the operands are stored in 16 bits and the arithmetic is fp32; here
 * storage and arithmetic are both fp32, the parity path for fp32 inputs.
 * Arguments as mha_fwd, with Q, K, V, O float [B, H, S, D].  D : 64 or 128.
 */
int mha_fwd_f32(const float* Q, const float* K, const float* V, float* O, float* LSE,
                int B, int H, int S, int D, float scale, int causal, void* stream);

/*
 * Single-query decode ("mmha"): for every sequence b and head h one query
 * attends to all cached keys of sequence b.  Page 3, sections 2.1-2.2 (one
 * query row against a K tile, fused GEMV + softmax), with the key range split
 * across thread blocks and merged with a log-sum-exp combine, the
 * cross-block normalisation that page 1 section 2.2 warns must not be done
 * per block.
 *
 *   q       : const bf16 [B, H, D].
 *   Kcache,
 *   Vcache  : const bf16 [sum_b seqlens[b], H, D]: the sequences packed back
 *             to back, token t of sequence b at row (sum_{b'<b} seqlens[b'] + t).
 *   seqlens : const int32 [B] in DEVICE memory, each >= 0; a sequence of length
 *             0 gets O = 0.
 *   O       : bf16 [B, H, D], written.
 *   B, H    : >= 1.  D : 64 or 128.  scale as in mha_fwd.
 *
 * Scratch: the partial results of the key splits (B*H*nsplit*(D+2) floats)
 * are allocated and freed stream-ordered on `stream` (cudaMallocAsync /
 * cudaFreeAsync from the device's default memory pool) inside the call.
 */
int mha_decode(const void* q, const void* Kcache, const void* Vcache, const int* seqlens,
               void* O, int B, int H, int D, float scale, void* stream);

/*
 * mha_decode on f16 data: q, Kcache, Vcache and O are f16 with the layouts
 * above; everything else (seqlens, scratch, asynchrony, errors) as mha_decode.
 */
int mha_decode_f16(const void* q, const void* Kcache, const void* Vcache, const int* seqlens,
                   void* O, int B, int H, int D, float scale, void* stream);

/*
 * mha_decode / mha_decode_f16 with the number of key splits chosen by the
 * caller.  The split count changes only how the keys of a row are divided
 * among thread blocks before the log-sum-exp merge (page 1, "Week 4 CUDA
 * notes", section 2.2: the blocks' normalisations are reconciled, never
 * applied per block), so every split count gives the same attention up to
 * fp32 rounding; this call lets a caller (or a test) pick it.
 *
 *   nsplit : 0 = the automatic choice of mha_decode (mha_decode_num_splits);
 *            1..64 = that many splits (1 = one block per row, no merge
 *            kernel, no scratch).  Other values: MHA_ERR_INVALID_ARG.
 *   dtype  : 0 = bf16, 1 = f16 (q, Kcache, Vcache and O); others
 *            MHA_ERR_UNSUPPORTED.
 *   other arguments, scratch and errors as mha_decode.
 */
int mha_decode_ex(const void* q, const void* Kcache, const void* Vcache, const int* seqlens,
                  void* O, int B, int H, int D, float scale, int nsplit, int dtype,
                  void* stream);

/*
 * mha_decode without allocating anything.  This entry point has no
 * counterpart on the pages the method comes from; it exists for callers
 * that cannot allocate device memory when they call: a serving loop that
 * plans all of its device memory up front and treats any later allocation
 * as an error, a device or driver mode without memory-pool support (where
 * the cudaMallocAsync that mha_decode uses fails), or code running while its
 * process's own allocator is busy.
 *
 * Arguments, layouts and results are those of mha_decode.  The split
 * partials go to one file-scope device array of
 * MHA_DECODE_NOALLOC_SCRATCH_BYTES (2 MiB) that every GPU which loads the
 * library holds until the process exits; the call itself makes no
 * cudaMalloc/cudaFree or other allocating call.  It uses mha_decode's split
 * count (mha_decode_num_splits) when the partials, B*H*splits*(D+2)*4
 * bytes, fit in the array, and otherwise the largest split count whose
 * partials fit, down to one split, which needs no scratch; the results
 * agree with mha_decode's to fp32 rounding (bit for bit when the split
 * count is the same).
 *
 * The first call in a CUDA context looks up the array's address in that
 * context (cudaGetSymbolAddress, with the device current) and keeps it
 * together with the context's unique ID; a call after the context was
 * destroyed and created again (cudaDeviceReset) looks it up again.  Make
 * the first call on a device, and the first after a reset, before any
 * stream capture.  All calls share the one array and it keeps
 * whatever the last call left there; no part of it has to start at zero,
 * since every slot a call reads was written earlier in that same call.
 * Calls that overlap on the GPU (for instance on two streams) race on the
 * array and may return wrong results: serialise them.
 */
#define MHA_DECODE_NOALLOC_SCRATCH_BYTES (2u * 1024u * 1024u)
int mha_decode_noalloc(const void* q, const void* Kcache, const void* Vcache,
                       const int* seqlens, void* O, int B, int H, int D, float scale,
                       void* stream);

/*
 * Number of key splits mha_decode uses for B sequences x H heads on the
 * current device (1 means no merge kernel and no scratch).  The scratch of
 * one mha_decode call is B*H*splits*(D+2)*4 bytes.  Returns <= 0 on a CUDA
 * error or an invalid argument.
 */
int mha_decode_num_splits(int B, int H);

/*
 * Which work-item schedule mha_fwd / mha_fwd_f16 (key_padding = 0) or the
 * _varlen calls (key_padding = 1) use for this shape: 1 = the wide groups
 * (about six 256-row query blocks per CTA per group of heads), 0 = the
 * narrow ones (about two).  A persistent grid of min(B*H*ceil(S/256),
 * sm_count) CTAs deals the query blocks; the choice is made per launch from
 * a model of each CTA's load (D = 64 and key padding always take the wide
 * groups).  sm_count <= 0 takes the current device's count.  Host
 * arithmetic only (no GPU work), except for reading the device's SM count.
 * Returns 1 or 0, or a negative MHA_ERR_* code: -MHA_ERR_INVALID_ARG for a
 * non-positive size or D other than 64 and 128, -MHA_ERR_CUDA when the SM
 * count cannot be read.
 */
int mha_prefill_wide_schedule(int B, int H, int S, int D, int causal, int key_padding,
                              int sm_count);

/*
 * The work items of one CTA of the same launch, in the order it takes them:
 * item i is the 256-row query block qp_out[i] (rows 256*qp .. 256*qp + 255)
 * of head row bh_out[i] = b*H + h.  The grid is min(B*H*ceil(S/256),
 * sm_count) CTAs and every (bh, qp) belongs to exactly one of them.
 *
 *   cta      : CTA index; outside [0, grid) the CTA has no items.
 *   bh_out, qp_out : host int arrays of `capacity` entries (caller-owned;
 *              may be NULL when capacity is 0); the first min(count,
 *              capacity) items are written.
 *   sm_count : as for mha_prefill_wide_schedule.
 *
 * Returns the CTA's item count (which may exceed capacity; call with
 * capacity 0 to size the arrays), or a negative MHA_ERR_* code:
 * -MHA_ERR_INVALID_ARG for a non-positive size, D other than 64 and 128,
 * B*H*S*D >= 2^31, a negative capacity or NULL arrays with capacity > 0;
 * -MHA_ERR_CUDA when the SM count cannot be read.  Host arithmetic only.
 */
int mha_prefill_schedule(int B, int H, int S, int D, int causal, int key_padding, int sm_count,
                         int cta, int* bh_out, int* qp_out, int capacity);

/*
 * Fused Q, K, V projection feeding the attention calls: page 3 section 2
 * (Q = X W_Q, K = X W_K, V = X W_V) with its section 2.1 shapes, the three
 * products fused into one GEMM as page 1 section 2.1 ("Week 4 CUDA notes")
 * does.  bf16 in and out, fp32 accumulation on the tensor cores.
 *
 *   X       : const bf16 [B, S, hidden] (row-major [B*S][hidden]).
 *   W       : const bf16 [hidden, 3*H*D] = [W_Q | W_K | W_V] (row-major).
 *   Q, K, V : bf16 [B, H, S, D], written: Q[b][h][s][d] = sum_k X[b][s][k] *
 *             W[k][h*D + d]; K uses columns H*D + h*D + d, V 2*H*D + h*D + d.
 *             This is the layout mha_fwd reads.
 *   hidden  : >= 1 and a multiple of 8.   D : 64 or 128.
 *   B*S*hidden, hidden*3*H*D and B*S*3*H*D each < 2^31.
 */
int mha_qkv_proj(const void* X, const void* W, void* Q, void* K, void* V, int B, int S,
                 int hidden, int H, int D, void* stream);

/*
 * Output projection after attention (page 1 section 2.1 lists it as one more
 * GEMM): the heads of O are concatenated, feature h*D + d of row (b, s) being
 * O[b][h][s][d], and multiplied by W_O.  This is also the per-head grouped
 * form Y = sum_h O_h W_O[h*D:(h+1)*D], summed in one fp32 accumulator.
 * bf16 in and out, tensor cores.
 *
 *   O       : const bf16 [B, H, S, D] (the layout mha_fwd writes).
 *   W       : const bf16 [H*D, n_out], row-major.
 *   Y       : bf16 [B, S, n_out], row-major, written.
 *   D : 64 or 128.   n_out : >= 1 and a multiple of 32.
 *   B*S*H*D, H*D*n_out and B*S*n_out each < 2^31.
 */
int mha_out_proj(const void* O, const void* W, void* Y, int B, int H, int S, int D, int n_out,
                 void* stream);

/*
 * The prefill of mha_fwd / mha_fwd_f16 / mha_fwd_varlen(_f16) behind one
 * entry point, with a choice of O's layout.
 *
 *   dtype    : 0 = bf16, 1 = f16 (Q, K, V and O).
 *   key_lens : as in mha_fwd_varlen, or NULL for no key padding.
 *   o_layout : 0 = O as [B, H, S, D] (as mha_fwd);
 *              1 = O as [B, S, H, D]: row (b, s) holds the heads of position s
 *              side by side (feature h*D + d), the concatenation the output
 *              projection multiplies by W_O (page "Week 4 CUDA notes"
 *              section 2.1), so that product reads O as a plain row-major
 *              [B*S, H*D] matrix (mha_out_proj_ex with o_layout 1).
 *   Q, K, V, LSE, sizes, scale, causal and errors as mha_fwd; an unknown
 *   dtype or o_layout returns MHA_ERR_UNSUPPORTED.
 */
int mha_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE,
               const int* key_lens, int B, int H, int S, int D, float scale, int causal,
               int dtype, int o_layout, void* stream);

/*
 * mha_out_proj with a choice of O's layout: o_layout 0 reads O as
 * [B, H, S, D] (as mha_out_proj), 1 reads O as [B, S, H, D], the row-major
 * [B*S, H*D] matrix of concatenated heads (what mha_fwd_ex writes with
 * o_layout 1).  Y, W, sizes and errors as mha_out_proj; the sums are taken in
 * the same order either way, so both layouts give the same Y bit for bit.
 */
int mha_out_proj_ex(const void* O, const void* W, void* Y, int B, int H, int S, int D, int n_out,
                    int o_layout, void* stream);

/*
 * Synchronises `stream`, then reads and clears the device error words that
 * bounded waits set (each with one atomic exchange on the device, in order
 * on `stream`, so a timeout recorded meanwhile by a launch on another stream
 * is kept for the next call rather than lost).  Returns MHA_OK,
 * MHA_ERR_TIMEOUT when a wait in some kernel of this library ran out since
 * the last call, or MHA_ERR_CUDA when the synchronisation itself failed.
 */
int mha_get_device_status(void* stream);

/* Static, human-readable text for an mha_status value. */
const char* mha_status_string(int status);

/* The cudaError_t value of the last call that returned MHA_ERR_CUDA (0 if none). */
int mha_last_cuda_error(void);

/*
 * Failure-detection hook: sets the time limit, in nanoseconds, of every
 * bounded device wait in later launches (default 2e9 = 2 s; 0 restores the
 * default).  A tiny limit makes waits run out on purpose so that the
 * timeout path — error word set, in-flight copies drained, tensor memory
 * freed, kernel returns — can be exercised without hanging anything.
 * Returns the previous limit.
 */
uint64_t mha_set_wait_limit_ns(uint64_t limit_ns);

/*
 * Failure-detection hook: mode 1 makes later mha_fwd launches withhold one
 * internal signal (each CTA's first "probabilities ready" arrival), a signal
 * that then never comes, so the bounded wait for it runs out; the kernel
 * records MHA_ERR_TIMEOUT, lets its in-flight copies and tensor-core work
 * finish, frees its tensor memory and returns.  Outputs of such a launch are
 * undefined.  Mode 0 (the default) turns it off.  Returns the previous mode,
 * or -1 for an unknown mode.
 */
int mha_set_fault_injection(int mode);

#ifdef __cplusplus
}
#endif

#endif /* MHA_GB300_H */
