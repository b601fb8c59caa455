/*
 * attnbwd.h: C ABI of the GB300 (sm_103a) attention backward library.
 *
 * The library computes the exact gradient of standard attention without
 * ever storing the N x N probability matrix: the backward recomputes
 * S = tau Q K^T and P = exp(S - LSE) tile by tile from the row statistic LSE
 * saved by the forward.
 *
 * Sources (web pages, cited by title and section):
 *   [FA-v1-bwd] "解析 FlashAttention（3）：FlashAttention-v1 反向传播",
 *               §1.1, §2.2-2.7 (eq. 1-8), §3 (eq. 9-16), §4 (Algorithm 4).
 *   [bwd-detail] "反向传播算法详解" (Inference Cookbook), §1.2-1.3
 *               (recompute, saved tensors), §2.1 (five gradients, dPsum,
 *               softcap), §3 (N-outer / Q-inner loop), §6 (dQ accumulation),
 *               §8.5 (GQA group sums).
 *
 * Conventions shared by every call
 * --------------------------------
 *  * Pointers are DEVICE pointers into memory the caller owns; the library
 *    never allocates or frees caller memory.
 *  * Layout is contiguous row-major: Q, O, dO, dQ and the dQ accumulator are
 *    [B, H, N, d]; K, V, dK, dV are [B, H_kv, N, d]; LSE and D are [B, H, N].
 *    bf16 tensors are passed as `void*` (IEEE bfloat16 bit patterns).
 *  * Query head h uses KV head h / (H / H_kv) (H must be a multiple of H_kv).
 *  * d must be 64 or 128 for the allocation-free backward; 64, 128 or 256
 *    for every other forward and backward call (attn_fwd, attn_fwd_ref and
 *    their local and dropout forms, attn_bwd, attn_bwd_local,
 *    attn_bwd_dropout, attn_bwd_deterministic, attn_bwd_finalize_partials);
 *    preprocess and finalize accept any d that is a multiple of 4. Other
 *    values return ATTN_ERR_UNSUPPORTED.
 *  * Every pointer must be 16-byte aligned (the kernels use TMA and 16-byte
 *    vector accesses).
 *  * `scale` is tau (usually 1/sqrt(d)); the logit is tau * q.k.
 *  * `softcap` > 0 enables the softcap: logit = c * tanh(tau q.k / c), whose
 *    derivative (1 - tanh^2) multiplies dS ([bwd-detail] §2.1(3)).
 *    softcap <= 0 disables it.
 *  * `causal` != 0 applies the lower-triangular mask: key j is visible to
 *    query i iff j <= i (queries and keys share the length N).
 *  * `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Every call is asynchronous on that stream.
 *  * Return value: ATTN_OK (0) or a negative ATTN_ERR_* code. Arguments are
 *    validated before anything is launched, so an error return means nothing
 *    was enqueued. B, H or N equal to 0 is a valid empty problem (no launch).
 *  * No exception crosses this interface. The library keeps one small
 *    device status word (see attn_device_status) and, for
 *    attn_bwd_noalloc, one fixed scratch array; it caches nothing else.
 */
#ifndef ATTNBWD_H_
#define ATTNBWD_H_

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_OK 0
#define ATTN_ERR_NULL (-1)           /* a required pointer is NULL */
#define ATTN_ERR_SHAPE (-2)          /* negative size, H % H_kv != 0, bad scale ... */
#define ATTN_ERR_UNSUPPORTED (-3)    /* head dimension not supported by this call */
#define ATTN_ERR_ALIGN (-4)          /* a pointer is not 16-byte aligned */
#define ATTN_ERR_LAUNCH (-5)         /* CUDA reported an error at launch */
#define ATTN_ERR_DEVICE_TIMEOUT (-6) /* a kernel gave up waiting (device status) */
#define ATTN_ERR_DEVICE (-7)         /* a kernel detected an internal fault */
#define ATTN_ERR_TOO_LARGE (-8)      /* a size exceeds what the kernels index */

/*
 * attn_fwd_ref: simple GPU forward producing the tensors the backward needs
 * ([bwd-detail] §1.3 saved-tensor table; [FA-v1-bwd] §1.1):
 *   S = tau Q K^T (softcap, causal mask), LSE_i = ln sum_j exp(S_ij),
 *   O = softmax(S) V.
 * In:  q [B,H,N,d] bf16, k, v [B,H_kv,N,d] bf16.
 * Out: o [B,H,N,d] bf16 (overwritten), lse [B,H,N] fp32 natural log
 *      (overwritten).
 * Arithmetic is fp32 with accurate exp/log/tanh; it is a reference-quality
 * producer of O and LSE, not a tuned kernel.
 */
int attn_fwd_ref(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int H_kv, int N, int d, float scale, int causal, float softcap, void* stream);

/*
 * Dropout ([FA-v1-bwd] §3.3 and Algorithm 4 of §4), drop probability
 * p_drop in [0, 1) (0 = none) and a 64-bit seed. Element (query i, key j) of
 * query head bh = b * H + h is kept iff word (i mod 4) of
 * Philox4x32-10(counter = (floor(i / 4), j, bh, 0), key = (seed mod 2^32,
 * seed >> 32)) is >= round(p_drop * 2^32) (Philox4x32-10: Salmon et al.,
 * "Parallel random numbers: as easy as 1, 2, 3", SC 2011); kept elements of
 * P are scaled by 1 / (1 - p_drop). LSE is that of P before dropout.
 *
 * attn_fwd_ref_dropout: attn_fwd_ref with dropout: O = (P o Z / (1 - p)) V.
 * attn_bwd_dropout: attn_bwd for that forward (same mask from the same
 *   seed): dV = (P o Z / (1 - p))^T dO, dP = (dO V^T) o Z / (1 - p),
 *   dS = P o (dP - D) with D = rowsum(dO o O) of the dropped O. Run it with
 *   attn_bwd_preprocess and attn_bwd_finalize as attn_bwd.
 * Both return ATTN_ERR_SHAPE for p_drop outside [0, 1).
 */
int attn_fwd_ref_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int H_kv, int N, int d, float scale, int causal,
                         float softcap, float p_drop, unsigned long long seed, void* stream);
int attn_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, float* dq_accum, void* dk, void* dv, int B, int H,
                     int H_kv, int N, int d, float scale, int causal, float softcap,
                     const float* dpsum, float p_drop, unsigned long long seed, void* stream);

/*
 * attn_fwd_dropout: attn_fwd (the one-pass tensor-core forward; scale > 0)
 * with the same dropout as attn_fwd_ref_dropout: O = (P o Z / (1 - p)) V with
 * the keep mask Z defined above, LSE that of P. One Philox call still serves
 * four elements: the four query rows of a call sit in four adjacent lanes,
 * each lane draws the call of one key and a shuffle transpose hands every
 * lane its own row's words.
 */
int attn_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int H_kv, int N, int d, float scale, int causal, float softcap,
                     float p_drop, unsigned long long seed, void* stream);

/*
 * attn_fwd: the same forward as attn_fwd_ref (same arguments, outputs and
 * layouts) on the tcgen05 tensor cores, in one pass with the online softmax
 * ([bwd-detail] §1.2; [FA-v1-bwd] §1.1 forward, §3.2 eq. 9-12 running
 * statistics): a CTA walks the visible key blocks of its queries once; O
 * accumulates un-normalised in fp32 tensor memory, rescaled only when a row
 * maximum grows by more than 2^8, and is divided by the row sum at the end.
 * P enters the PV GEMM as bf16. One CTA per SM walks blocks of 128 queries
 * (persistent, heaviest first); a block's key blocks alternate between two S
 * buffers and its keys are split between two softmax warpgroups, and the
 * next block's loads overlap the current one's last GEMMs and epilogue.
 * scale must be > 0 (ATTN_ERR_SHAPE otherwise).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int H_kv, int N, int d, float scale, int causal, float softcap, void* stream);

/*
 * Local (sliding-window) attention ([bwd-detail] §3.4, the third masking
 * phase of the Q-inner loop: query blocks at the window's edge are masked
 * elementwise, those inside it run unmasked, those outside it are skipped).
 * Key j is visible to query i iff
 *     i - window_left <= j <= i + window_right,
 * and, if causal != 0, also j <= i. A negative bound (or one of N or more)
 * leaves that side unbounded, so (-1, -1) is the plain call, and (-1, 0)
 * without causal equals the causal mask. Every row keeps its own key (the
 * diagonal), so LSE is always finite.
 *
 * attn_fwd_local, attn_fwd_ref_local: attn_fwd / attn_fwd_ref under that
 *   mask (same outputs and layouts).
 * attn_bwd_local: attn_bwd under that mask; a CTA visits only the query
 *   blocks of its key block's band. Run it with attn_bwd_preprocess and
 *   attn_bwd_finalize as attn_bwd.
 * Arguments, errors and stream order as for the calls they extend.
 */
int attn_fwd_local(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int H_kv, int N, int d, float scale, int causal, float softcap,
                   int window_left, int window_right, void* stream);
int attn_fwd_ref_local(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int H_kv, int N, int d, float scale, int causal, float softcap,
                       int window_left, int window_right, void* stream);
int attn_bwd_local(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, float* dq_accum, void* dk, void* dv, int B, int H, int H_kv,
                   int N, int d, float scale, int causal, float softcap, const float* dpsum,
                   int window_left, int window_right, void* stream);

/*
 * attn_bwd_preprocess: D = rowsum(dO o O) ([FA-v1-bwd] §2.4 eq. 6;
 * [bwd-detail] §2.1(3), "dPsum", computed before the main kernel) and
 * dq_accum := 0.
 * In:  o, dO [B,H,N,d] bf16.
 * Out: dpsum [B,H,N] fp32 (overwritten); dq_accum [B,H,N,d] fp32 (zeroed;
 *      may be NULL, then only D is computed).
 */
int attn_bwd_preprocess(const void* o, const void* dO, float* dpsum, float* dq_accum, int B,
                        int H, int N, int d, void* stream);

/*
 * attn_bwd: main backward kernel, N-outer / Q-inner ([bwd-detail] §3,
 * [FA-v1-bwd] §4). One CTA owns 128 keys of one KV head, keeps dK and dV
 * in tensor memory while it walks every query block of every query head of
 * the group, and runs the five GEMMs per tile on the tensor cores:
 *   S^T = K Q^T, dP^T = V dO^T, P = exp(S - LSE), dS = P o (dP - D)
 *   [o (1 - tanh^2)], dV += P^T dO, dK += dS^T Q, dQ_partial = dS K.
 * In:  q, o, dO [B,H,N,d] bf16; k, v [B,H_kv,N,d] bf16; lse [B,H,N] fp32
 *      (natural log, from the forward); dpsum [B,H,N] fp32 (from
 *      attn_bwd_preprocess).
 * In/out: dq_accum [B,H,N,d] fp32: partial dQ (without the factor tau) is
 *      ADDED with fp32 atomics; it must be zeroed first (preprocess does).
 * Out: dk, dv [B,H_kv,N,d] bf16, overwritten; dk includes tau; for H_kv < H
 *      they are summed over the head group.
 * `o` is accepted for interface completeness; D already carries its use.
 * d = 256 runs a kernel of its own ([bwd-detail] §8.3 slices the d = 256
 * GEMMs): a CTA accumulates one half of d for 128 keys over query tiles of
 * 64, recomputing S and dP over the full d (seven GEMM-equivalents per tile
 * instead of five); dQ accumulates the same way. That kernel also serves
 * attn_bwd_local, attn_bwd_dropout and attn_bwd_deterministic at d = 256.
 * Order on the stream: attn_bwd_preprocess, attn_bwd, attn_bwd_finalize.
 * dQ is summed with fp32 atomics, so it may differ in the last bits from run
 * to run; dK and dV are summed on chip in a fixed order.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
             const float* lse, float* dq_accum, void* dk, void* dv, int B, int H, int H_kv, int N,
             int d, float scale, int causal, float softcap, const float* dpsum, void* stream);

/*
 * Deterministic dQ ([bwd-detail] §6.4: the fp32 atomics make dQ differ in the
 * last bits between runs; a fixed order of the additions removes that).
 *
 * attn_bwd_dq_partials_bytes: size of the partials workspace, in bytes, or a
 *   negative ATTN_ERR_* code: one fp32 tile of 128 rows x d per query head
 *   and (query block m, key block n) pair the mask keeps,
 *   B * H * P * 128 * d * 4 with P = M (M + 1) / 2 (causal) or M * M, and
 *   M = ceil(N / 128).
 * attn_bwd_deterministic: attn_bwd with the same arguments, except that each
 *   dQ tile (without the factor tau) is STORED into dq_partials (laid out as
 *   [B*H, P, 128, d], pair index m (m + 1) / 2 + n if causal, else m M + n)
 *   instead of being added into an accumulator; nothing needs zeroing
 *   (attn_bwd_preprocess may be called with dq_accum = NULL). dK, dV as in
 *   attn_bwd (already reproducible).
 * attn_bwd_finalize_partials: dq = bf16(scale * sum over n = 0, 1, ... of
 *   the partial tiles of each query block), always in that order, so dQ is
 *   identical bit for bit from run to run. `causal` must match the backward.
 * Order on the stream: attn_bwd_preprocess, attn_bwd_deterministic,
 * attn_bwd_finalize_partials. Costs one fp32 tile write and read per pair
 * (2.2 GB each way for B=2, H=32, N=4096, d=128 causal).
 */
long long attn_bwd_dq_partials_bytes(int B, int H, int N, int d, int causal);
int attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                           const void* dO, const float* lse, float* dq_partials, void* dk,
                           void* dv, int B, int H, int H_kv, int N, int d, float scale,
                           int causal, float softcap, const float* dpsum, void* stream);
int attn_bwd_finalize_partials(const float* dq_partials, void* dq, float scale, int B, int H,
                               int N, int d, int causal, void* stream);

/*
 * attn_bwd_finalize: dq = bf16(scale * dq_accum) ([FA-v1-bwd] eq. 7: the
 * factor tau of dQ = tau dS K is applied here).
 * In:  dq_accum [B,H,N,d] fp32.  Out: dq [B,H,N,d] bf16, overwritten.
 */
int attn_bwd_finalize(const float* dq_accum, void* dq, float scale, int B, int H, int N, int d,
                      void* stream);

/*
 * attn_bwd_noalloc: the whole backward (attn_bwd_preprocess, attn_bwd,
 * attn_bwd_finalize) in one call that allocates nothing. The pages have no
 * counterpart for it: it exists for callers that cannot allocate device
 * memory (graph-captured code where allocation is not allowed, plugins that
 * are handed fixed buffers, runtimes whose allocator must not be re-entered).
 * Arguments mean what they mean for attn_bwd; dq [B,H,N,d] bf16 receives the
 * finished dQ (tau applied), dk, dv as for attn_bwd.
 * Scratch: the fp32 dQ accumulator and D live in one file-scope device array
 * of 8,388,608 floats (32 MiB) that every device loading the library keeps
 * until the process exits. A problem needs B*H*N*d + B*H*N floats; larger
 * problems return ATTN_ERR_TOO_LARGE.
 * Every check of the three steps (pointers, shapes, d = 64 or 128, scale
 * finite and non-zero, softcap not NaN, 16-byte alignment of all nine
 * pointers, the size limit) runs before the first launch: an argument error
 * enqueues nothing and leaves the array untouched. Only ATTN_ERR_LAUNCH, an
 * error CUDA reports at a launch, can come after a step was enqueued.
 * All calls share that array: calls whose GPU work overlaps (unordered
 * streams, several host threads) race and give wrong results. The first call
 * on a device looks up the array's address with that device current; make it
 * before any stream capture.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int H_kv,
                     int N, int d, float scale, int causal, float softcap, void* stream);

/*
 * attn_device_status: waits for `stream`, then reads the library's device
 * status word into *status (0 = no fault; ATTN_ERR_DEVICE_TIMEOUT when a
 * kernel gave up waiting on a barrier; ATTN_ERR_DEVICE for an internal
 * check). clear != 0 resets it to 0. Returns ATTN_OK or a launch error.
 */
int attn_device_status(int* status, int clear, void* stream);

/*
 * attn_selftest_wait_timeout: runs, on `stream`, a one-block kernel that
 * takes the bounded mbarrier wait the backward kernels use on a barrier that
 * nothing arrives on, with a limit of about half a millisecond instead of
 * the kernels' one second. The wait gives up, raises the block's abort flag
 * (a second warp waiting on another barrier returns on it) and records
 * ATTN_ERR_DEVICE_TIMEOUT. The device status word is cleared first; on
 * return *status holds what the kernel recorded (ATTN_ERR_DEVICE_TIMEOUT
 * when the mechanism works) and the word is cleared again. Nothing faults
 * or traps, so the context stays usable. Returns ATTN_OK or a launch error.
 */
int attn_selftest_wait_timeout(int* status, void* stream);

/* Static description of an error code; never NULL. */
const char* attn_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* ATTNBWD_H_ */
