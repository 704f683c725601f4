/*
 * libssmverify -- the Mamba-layer step of speculative decoding, on one GPU.
 *
 * Source of the method: the paper "The Mamba in the Llama: Distilling and
 * Accelerating Hybrid Models" (Wang, Paliotta, May, Rush, Dao; abstract: a
 * hardware-aware speculative decoding algorithm for Mamba and hybrid models)
 * and its news summary "Llama 3+Mamba强强联手！蒸馏到RNN，推理速度提升1.6倍"
 * (speculative-decoding section: the draft model proposes K tokens, the Mamba
 * layers of the verifier run them one after another from the cached state,
 * accepted tokens advance the state without storing intermediate states, and
 * at the first wrong token the state rolls back to the last accepted one).
 *
 * The recurrence (the discrete-time linear RNN that the method overview says
 * Mamba's continuous-time SSM yields; zero-order hold on A, Euler on B), per
 * sequence b, head h (B/C group g = h / (nheads / ngroups)) and token t:
 *
 *     Abar_t      = exp(dt_t * A_h)
 *     h_t[p][n]   = Abar_t * h_{t-1}[p][n] + (dt_t * x_t[p]) * B_t[n]
 *     y_t[p]      = sum_n C_t[n] * h_t[p][n] + D_h * x_t[p]
 *
 * with C, B, x in the roles of attention's Q, K, V (the attention-to-RNN
 * correspondence the distillation's initialisation rests on).
 *
 * ------------------------------------------------------------------------
 * Layouts (row-major, contiguous, last index fastest):
 *
 *   state       float [batch][nheads][headdim][dstate]   cached h, fp32
 *   x           in_t  [batch][ntok][nheads][headdim]
 *   B, C        in_t  [batch][ntok][ngroups][dstate]
 *   dt          in_t  [batch][ntok][nheads]   already positive (no softplus)
 *   A, D        float [nheads]
 *   y           float [batch][ntok][nheads][headdim]
 *   accept_len  int32 [batch]    accepted draft tokens j in [0, ntok]
 *
 * in_t is float (SSM_F32) or bf16 (SSM_BF16), chosen by desc->in_dtype.
 *
 * Ownership and threading: every pointer is a DEVICE pointer owned by the
 * caller (for the whole time the launched work runs). The library allocates
 * nothing, frees nothing and never synchronises; the only state it keeps
 * between calls is a cache of immutable device properties (SM count and
 * resident blocks per SM, per kernel and device), so calls are thread-safe
 * (ssm_prefill_scratch alone also uses a fixed device array; see there).
 * Every entry point only validates its arguments and enqueues one kernel
 * (ssm_prefill: up to three; ssm_copy_from_host_n: one per segment when the
 * segments are not all 16-byte aligned) on `stream` (a cudaStream_t passed
 * as void*, NULL = the legacy default stream) on the current device. Calls
 * are asynchronous. ssm_copy_from_host and ssm_copy_from_host_n alone take
 * host pointers (their sources). Launches of the verify / commit kernel with
 * no more blocks than the device has SMs (a decode step of a few sequences)
 * use programmatic dependent launch: the kernel may become resident while the
 * previous kernel of the stream finishes, and waits for that kernel's
 * completion before touching memory, so stream order is kept.
 *
 * Errors: the return value is SSM_OK or an SSM_ERR_* code. Argument errors
 * are detected on the host before anything is launched (no device work is
 * enqueued then). SSM_ERR_CUDA reports a failed launch; the CUDA error code
 * of the calling thread's last failed launch is ssm_last_cuda_error().
 * Errors found on the device never trap. An accept_len outside [0, ntok]
 * leaves the affected sequence's state untouched and, if dev_status is not
 * NULL, ORs SSM_STATUS_BAD_ACCEPT_LEN into *dev_status. A kernel block whose
 * wait for its own state copy exceeds one second (which does not happen on a
 * healthy device) stops early and ORs SSM_STATUS_TIMEOUT: its outputs are
 * then incomplete. The caller reads *dev_status after its own
 * synchronisation; it is only ever OR-ed into, so the caller zeroes it.
 *
 * Supported shapes: dstate in {16, 32, 64, 128, 256}; any headdim >= 1;
 * nheads % ngroups == 0; ntok >= 1; batch >= 0 (batch == 0 is a no-op that
 * inspects no pointer). Alignment: state 16 bytes; x, B, C, dt their element
 * size; A, D, y, accept_len, dev_status 4 bytes. x whose base is 16-byte
 * aligned with headdim * element size a multiple of 16, and 16-byte aligned
 * B / C, are read with 128-bit loads; other layouts take a scalar path with
 * the same results.
 * Aliasing: a buffer the call writes (y; state for the committing calls) must
 * not overlap any other buffer of the call.
 */
#ifndef SSMVERIFY_H
#define SSMVERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSM_VERSION 1

/* element type of x, B, C, dt */
#define SSM_F32 0
#define SSM_BF16 1

/* return codes */
#define SSM_OK 0
#define SSM_ERR_NULL 1        /* a required pointer (or desc) is NULL */
#define SSM_ERR_SHAPE 2       /* a dimension is out of range, nheads % ngroups != 0, ntok < 1 ... */
#define SSM_ERR_UNSUPPORTED 3 /* dstate or in_dtype has no kernel */
#define SSM_ERR_ALIGN 4       /* a pointer is not aligned as required */
#define SSM_ERR_ALIAS 5       /* a written buffer overlaps another buffer */
#define SSM_ERR_CUDA 6        /* the kernel launch failed */

/* bits OR-ed into *dev_status by the device */
#define SSM_STATUS_BAD_ACCEPT_LEN 1u
#define SSM_STATUS_TIMEOUT 2u
#define SSM_STATUS_BAD_TOKEN 4u /* acceptance: a draft token outside [0, vocab) */
#define SSM_STATUS_BAD_SLOT 8u  /* pool: a sequence's slot outside [0, nslots) */

typedef struct {
    int32_t batch;    /* sequences */
    int32_t nheads;   /* H */
    int32_t headdim;  /* P */
    int32_t dstate;   /* N */
    int32_t ngroups;  /* G: B/C groups; head h uses group h / (H / G) */
    int32_t ntok;     /* K: draft tokens per sequence */
    int32_t in_dtype; /* SSM_F32 or SSM_BF16 for x, B, C, dt */
    int32_t nlayers;  /* layers in one call: 0 or 1 = one layer (the layouts above); L > 1: a layer stack */
} ssm_desc_t;

/*
 * Layer stacks (desc->nlayers = L > 1; ssm_verify, ssm_commit,
 * ssm_verify_commit, ssm_commit_verify, ssm_step and their pool variants).
 * A hybrid model runs the
 * same K draft tokens through every Mamba layer, each layer with its own
 * cached state and its own inputs (the speculative-decoding section: every
 * Mamba layer of the verifier rolls back to the same last accepted token).
 * One call then covers all L layers: state, x, B, C, dt, y (and x_prev,
 * B_prev, dt_prev) carry a leading [L] dimension in front of their layouts
 * above (state [L][batch][nheads][headdim][dstate], x [L][batch][ntok]
 * [nheads][headdim], ...), A and D are [L][nheads], and accept_len (and
 * accept_len_prev) stays [batch]: one accepted prefix per sequence, shared
 * by every layer. A pool is then [L][nslots][nheads][headdim][dstate] (layer
 * l's pool is states[l]) and slot[batch] maps a sequence to the same slot in
 * every layer. The result equals L single-layer calls on the slices. Prefill
 * takes one layer (L > 1 there: SSM_ERR_UNSUPPORTED). nlayers < 0:
 * SSM_ERR_SHAPE.
 */

/*
 * ssm_verify -- run the K draft tokens from the cached state and emit y for
 * every token; the state is only read. This is the verifier's Mamba-layer
 * pass over the draft (speculative-decoding section of the news summary);
 * y is produced for all K tokens because acceptance is decided from them.
 */
int ssm_verify(const ssm_desc_t *desc, const float *state, const void *x, const void *B, const void *C,
               const void *dt, const float *A, const float *D, float *y, uint32_t *dev_status, void *stream);

/*
 * ssm_commit -- advance each sequence's cached state by its accepted prefix:
 * replay tokens 0 .. j-1 (j = accept_len[b]) and write h_j in place; j = 0
 * leaves the state unchanged (the rollback to the last accepted token of the
 * speculative-decoding section). C, D and y are not used. An accept_len
 * outside [0, ntok] leaves that sequence untouched and sets a dev_status bit.
 */
int ssm_commit(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *dt,
               const float *A, const int32_t *accept_len, uint32_t *dev_status, void *stream);

/*
 * ssm_verify_commit -- ssm_verify and ssm_commit fused for callers that know
 * accept_len when they launch: one read of the state, y for all K tokens,
 * and one in-place write of h_j (no write when j = 0). No intermediate state
 * is stored. Same accept_len rules as ssm_commit.
 */
int ssm_verify_commit(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *C,
                      const void *dt, const float *A, const float *D, const int32_t *accept_len, float *y,
                      uint32_t *dev_status, void *stream);

/*
 * ssm_commit_verify -- the serving order, where accept_len is known only
 * after every layer has verified: commit the previous round's accepted
 * prefix and verify the new draft tokens in one pass over the state (one
 * read, one write). For each sequence, replay tokens 0 .. j-1 of the
 * previous round's block (x_prev / B_prev / dt_prev, laid out like x / B /
 * dt with prev_ntok tokens; j = accept_len_prev[b]), write h_j in place
 * (nothing when j = 0), then run the desc->ntok new draft tokens from h_j and
 * emit y for every one of them; the new drafts' states are not stored (they
 * are committed by the next call). The result equals ssm_commit(previous
 * block, accept_len_prev) followed by ssm_verify(new block), bit for bit.
 * This is the speculative-decoding section's accept / roll back / continue
 * loop with the state update deferred to the next round. An accept_len_prev
 * outside [0, prev_ntok] replays nothing and writes nothing for that
 * sequence (y is still produced) and sets SSM_STATUS_BAD_ACCEPT_LEN.
 * prev_ntok >= 1; the previous block must not overlap the written buffers.
 */
int ssm_commit_verify(const ssm_desc_t *desc, float *state, int32_t prev_ntok, const void *x_prev,
                      const void *B_prev, const void *dt_prev, const int32_t *accept_len_prev, const void *x,
                      const void *B, const void *C, const void *dt, const float *A, const float *D, float *y,
                      uint32_t *dev_status, void *stream);

/*
 * ssm_step -- plain decoding, one token (desc->ntok must be 1): y for the
 * token and the state advanced by it in place. This is the ordinary decoding
 * that speculative decoding is compared against (results section of the news
 * summary).
 */
int ssm_step(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *C,
             const void *dt, const float *A, const float *D, float *y, uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * State pool (serving) and prefill.
 *
 * A serving loop keeps the cached states of its live sequences in a pool and
 * runs each step on whichever sequences are scheduled: sequence b of a call
 * uses pool slot slot[b]. The pool variants below are the entry points
 * above with `state` replaced by a pool; everything else (layouts of the
 * inputs and y, accept_len, errors) is unchanged. A slot outside
 * [0, nslots) leaves that sequence's y and state unwritten and ORs
 * SSM_STATUS_BAD_SLOT into *dev_status. Two sequences of one call must not
 * share a slot (their updates would race; nothing checks this on the device).
 *
 * Prefill runs a prompt through the layer and leaves the state at its last
 * token in the cache: the state the speculative rounds start from (the
 * speculative-decoding section's cached state; the method overview's
 * recurrence applied token after token). It equals ssm_verify_commit with
 * every token accepted; for long prompts on few sequences it splits the
 * prompt into chunks and runs them side by side (each chunk's state from
 * h = 0, a scan that carries the state across the chunks, then every chunk's
 * outputs from the state it starts from), which regroups the same
 * recurrence and agrees with it to fp32 rounding.
 * ------------------------------------------------------------------------ */

typedef struct {
    float *states;        /* [nslots][nheads][headdim][dstate] fp32 ([nlayers][nslots]... for a layer stack), 16-byte aligned */
    const int32_t *slot;  /* [batch] slot of each sequence, device memory; NULL: sequence b uses slot b */
    int32_t nslots;       /* >= 1; >= batch when slot is NULL */
    int32_t reserved;     /* must be 0 */
} ssm_pool_t;

int ssm_verify_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *C,
                    const void *dt, const float *A, const float *D, float *y, uint32_t *dev_status, void *stream);
int ssm_commit_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *dt,
                    const float *A, const int32_t *accept_len, uint32_t *dev_status, void *stream);
int ssm_verify_commit_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B,
                           const void *C, const void *dt, const float *A, const float *D, const int32_t *accept_len,
                           float *y, uint32_t *dev_status, void *stream);
int ssm_commit_verify_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, int32_t prev_ntok, const void *x_prev,
                           const void *B_prev, const void *dt_prev, const int32_t *accept_len_prev, const void *x,
                           const void *B, const void *C, const void *dt, const float *A, const float *D, float *y,
                           uint32_t *dev_status, void *stream);
int ssm_step_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *C,
                  const void *dt, const float *A, const float *D, float *y, uint32_t *dev_status, void *stream);

/*
 * ssm_prefill_workspace_bytes -- device workspace that ssm_prefill would use
 * for this shape on the current device (0: it runs in one pass and needs
 * none): batch * (ntok / L) states for the chunk length L it picks, plus a
 * small map of the chunks' slots (4 bytes per chunk) and each chunk's decay
 * product per head (4 bytes per chunk and head), each rounded up to 16 bytes.
 * L = 128 for bf16 inputs with dstate 128, headdim a multiple of 64 and
 * ntok a multiple of 128 of at least 256 (the tensor-core chunk passes);
 * other shapes chunk only when one pass would not fill the device, with the
 * largest L of 128, 64, 32, 16 that divides ntok into at least two chunks and
 * gives a full wave of tiles (else the smallest that divides it).
 */
int64_t ssm_prefill_workspace_bytes(const ssm_desc_t *desc);

/*
 * ssm_prefill -- run desc->ntok prompt tokens of every sequence from its
 * cached state (pool slot; zero it first for a fresh prompt), write y for
 * every token and leave the state after the last token in the slot. x, B, C,
 * dt, y have the layouts above with ntok = prompt length. `workspace`
 * (device, 16-byte aligned, workspace_bytes long; may be NULL) lets the
 * prompt be chunked; with too little workspace the call takes the one-pass
 * form (same results to rounding). The workspace must not overlap any other
 * buffer. Launches up to three kernels on `stream`.
 */
int ssm_prefill(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *C,
                const void *dt, const float *A, const float *D, float *y, void *workspace, int64_t workspace_bytes,
                uint32_t *dev_status, void *stream);

/*
 * ssm_prefill_scratch -- ssm_prefill without a caller workspace: the chunked
 * form runs in a fixed device array of SSM_PREFILL_SCRATCH_BYTES inside the
 * library (part of the library's device code: each CUDA context that loads
 * the library holds one copy until it is destroyed). The
 * chunk length is chosen among those whose workspace fits in the array;
 * where none fits the one-pass form runs (it needs no workspace, but takes
 * the prompt token after token), so results equal ssm_prefill's with a
 * workspace of SSM_PREFILL_SCRATCH_BYTES. Nothing in the array needs to start
 * at zero. Calls in the same CUDA context that may overlap on the device
 * (issued on other streams, from other host threads, or while an earlier
 * call still runs on another stream) race on the array: order them on one
 * stream. (Each context has its own copy of the array.) The array's device
 * address is looked up on every call, so the call stays correct after
 * cudaDeviceReset. The pages have no counterpart; this exists for callers
 * that cannot allocate device memory: a host runtime that owns every device
 * allocation itself and hands this library only its tensors' pointers, or a
 * latency-critical serving loop that must not enter cudaMalloc (which can
 * synchronise the device) between steps.
 */
#define SSM_PREFILL_SCRATCH_BYTES (64ll << 20)
int ssm_prefill_scratch(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *C,
                        const void *dt, const float *A, const float *D, float *y, uint32_t *dev_status, void *stream);

/*
 * ssm_selftest_wait_timeout -- failure-detection self-test of the bounded
 * waits the kernels use for their bulk copies (every such wait gives up after
 * about one second and reports SSM_STATUS_TIMEOUT instead of hanging). It
 * launches one warp that waits on a transaction that is announced but never
 * delivered (no copy is issued), so the wait runs out: after about one second
 * SSM_STATUS_TIMEOUT is OR-ed into *dev_status (required, 4-byte aligned
 * device word). Nothing else is touched and the device stays usable.
 */
int ssm_selftest_wait_timeout(uint32_t *dev_status, void *stream);

/* ------------------------------------------------------------------------
 * Acceptance of draft tokens (the step right after the verifier's pass).
 *
 * Source: the speculative-decoding section of the news summary (the draft
 * proposes K tokens; tokens the verifier agrees with are accepted; at the
 * first it does not, the remaining drafts are dropped and the state rolls
 * back to the last accepted token; with all K accepted the next round
 * starts) and the method overview of "The Mamba in the Llama", which calls
 * the procedure a speculative sampling algorithm. accept_len is written to
 * device memory in the layout ssm_commit / ssm_verify_commit /
 * ssm_commit_verify read, so acceptance needs no trip through the host.
 *
 * Layouts (row-major, contiguous):
 *   target_logits  logit_t [batch][ntok + 1][vocab]  verifier logits at every
 *                  draft position and at the bonus position ntok
 *   draft_logits   logit_t [batch][ntok][vocab]      draft-model logits
 *   draft_tokens   int32   [batch][ntok]
 *   uniform        float   [batch][ntok + 1]          U[0, 1) draws (sampling)
 *   accept_len     int32   [batch]   out: j in [0, ntok]
 *   next_token     int32   [batch]   out: the token that follows the accepted
 *                  prefix (a correction after a rejection, the bonus token
 *                  when j = ntok)
 * logit_t is float (SSM_F32) or bf16 (SSM_BF16). Every row must hold at least
 * one finite logit; NaN logits give unspecified results.
 *
 * Precision: probabilities are fp32 (exp(l - max) with subnormal results
 * flushed to zero, divided by the row's sum). Sums run in an order of the
 * library's choosing, so a decision whose threshold lies within fp32 rounding
 * of the drawn uniform may go either way; the bound is about 3e-5 relative
 * for an acceptance ratio and about 3e-5 of the summed probability mass for
 * the next-token threshold.
 *
 * Alignment: logits their element size (16-byte aligned logits with
 * vocab * element size a multiple of 16 take 128-bit loads; others a scalar
 * path with the same results); the int32 / float arrays and dev_status 4
 * bytes. Outputs must not overlap inputs or each other. A draft token outside
 * [0, vocab) counts as a rejection at its position (the next token is then
 * drawn from, or is the most likely token of, the verifier's distribution
 * there) and ORs SSM_STATUS_BAD_TOKEN into *dev_status.
 * ------------------------------------------------------------------------ */

#define SSM_ACCEPT_MAX_NTOK 32
#define SSM_ACCEPT_MAX_VOCAB (1 << 28)

typedef struct {
    int32_t batch;       /* sequences (0 is a no-op) */
    int32_t ntok;        /* K: draft tokens per sequence, 1 .. SSM_ACCEPT_MAX_NTOK */
    int32_t vocab;       /* V: 1 .. SSM_ACCEPT_MAX_VOCAB */
    int32_t logit_dtype; /* SSM_F32 or SSM_BF16 */
} ssm_accept_desc_t;

/*
 * ssm_accept_greedy -- accept draft token t while it is the verifier's most
 * likely token at position t (ties go to the smallest token index);
 * next_token is the verifier's most likely token at j = accept_len.
 */
int ssm_accept_greedy(const ssm_accept_desc_t *desc, const void *target_logits, const int32_t *draft_tokens,
                      int32_t *accept_len, int32_t *next_token, uint32_t *dev_status, void *stream);

/*
 * ssm_accept_sample -- speculative sampling: with p_t = softmax(target row t)
 * and q_t = softmax(draft row t), accept draft token x_t while
 * uniform[t] < p_t(x_t) / q_t(x_t) (always when q_t(x_t) = 0). At the first
 * rejection j < ntok the next token is drawn from the normalised residual
 * max(0, p_j - q_j), after ntok acceptances from p_ntok: the smallest index
 * whose cumulative weight exceeds uniform[ntok] times the total weight (the
 * last index of positive weight if rounding leaves none; vocab - 1 if no
 * weight is positive).
 */
int ssm_accept_sample(const ssm_accept_desc_t *desc, const void *target_logits, const void *draft_logits,
                      const int32_t *draft_tokens, const float *uniform, int32_t *accept_len, int32_t *next_token,
                      uint32_t *dev_status, void *stream);

/*
 * ssm_copy_from_host -- copy `bytes` from page-locked host memory `src` to
 * device memory `dst` with the SMs reading the host memory through its
 * unified address (16-byte vectors where both are 16-byte aligned), enqueued
 * on `stream` like a kernel. For the host front end: on B300 machines this
 * moves megabyte-sized step inputs at 35-37 GB/s where the copy engines
 * reach 12-14 GB/s. `src` must be page-locked (cudaHostAlloc /
 * cudaHostRegister) and `dst` device memory, else SSM_ERR_UNSUPPORTED is
 * returned before anything is launched; overlapping ranges give
 * SSM_ERR_ALIAS. The pages have no counterpart (a data-movement helper).
 */
int ssm_copy_from_host(void *dst, const void *src, int64_t bytes, void *stream);

/*
 * ssm_copy_from_host_n -- several such copies in one launch: segment i copies
 * segs[i].bytes from page-locked host memory segs[i].src to device memory
 * segs[i].dst. A step's inputs (x, B, C, dt, accept_len of a sequence chunk)
 * then cost one launch instead of one per tensor. `segs` is a host array of
 * 0 <= nseg <= SSM_COPY_MAX_SEGMENTS entries, read before the call returns.
 * Per segment the rules of ssm_copy_from_host apply; in addition no two
 * segments' destinations, and no destination and source, may overlap
 * (SSM_ERR_ALIAS). Where every segment's source and destination are 16-byte
 * aligned a single kernel copies them all; otherwise each segment takes its
 * own ssm_copy_from_host.
 */
#define SSM_COPY_MAX_SEGMENTS 8
typedef struct {
    void *dst;        /* device memory */
    const void *src;  /* page-locked host memory */
    int64_t bytes;    /* >= 0 */
} ssm_copy_segment_t;
int ssm_copy_from_host_n(const ssm_copy_segment_t *segs, int32_t nseg, void *stream);

/* A static, human-readable string for an SSM_* return code. */
const char *ssm_strerror(int code);

/* The CUDA error (cudaError_t as int) of this thread's last failed launch, 0 if none. */
int ssm_last_cuda_error(void);

/* SSM_VERSION of the built library. */
int ssm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SSMVERIFY_H */
