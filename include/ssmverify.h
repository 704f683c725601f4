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
 * nothing, frees nothing, never synchronises and keeps no mutable global
 * state; every entry point only validates its arguments and enqueues one
 * kernel on `stream` (a cudaStream_t passed as void*, NULL = the legacy
 * default stream) on the current device. Calls are asynchronous.
 *
 * Errors: the return value is SSM_OK or an SSM_ERR_* code. Argument errors
 * are detected on the host before anything is launched (no device work is
 * enqueued then). SSM_ERR_CUDA reports a failed launch; the CUDA error code
 * of the calling thread's last failed launch is ssm_last_cuda_error().
 * Errors found on the device (an accept_len outside [0, ntok]) never trap:
 * the affected sequence's state is left untouched and, if dev_status is not
 * NULL, SSM_STATUS_BAD_ACCEPT_LEN is OR-ed into *dev_status, which the caller
 * reads after its own synchronisation.
 *
 * Supported shapes: dstate in {16, 32, 64, 128, 256}; any headdim >= 1;
 * nheads % ngroups == 0; ntok >= 1; batch >= 0 (batch == 0 is a no-op that
 * inspects no pointer). Alignment: state 16 bytes; x, B, C, dt their element
 * size; A, D, y, accept_len, dev_status 4 bytes.
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

typedef struct {
    int32_t batch;    /* sequences */
    int32_t nheads;   /* H */
    int32_t headdim;  /* P */
    int32_t dstate;   /* N */
    int32_t ngroups;  /* G: B/C groups; head h uses group h / (H / G) */
    int32_t ntok;     /* K: draft tokens per sequence */
    int32_t in_dtype; /* SSM_F32 or SSM_BF16 for x, B, C, dt */
    int32_t reserved; /* must be 0 */
} ssm_desc_t;

/*
 * ssm_verify -- run the K draft tokens from the cached state and emit y for
 * every token; the state is only read. This is the verifier's Mamba-layer
 * pass over the draft (speculative-decoding section of the news summary);
 * y is produced for all K tokens because acceptance is decided from them.
 */
int ssm_verify(const ssm_desc_t *desc, const float *state, const void *x, const void *B, const void *C,
               const void *dt, const float *A, const float *D, float *y, void *stream);

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
 * ssm_step -- plain decoding, one token (desc->ntok must be 1): y for the
 * token and the state advanced by it in place. This is the ordinary decoding
 * that speculative decoding is compared against (results section of the news
 * summary).
 */
int ssm_step(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *C,
             const void *dt, const float *A, const float *D, float *y, void *stream);

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
