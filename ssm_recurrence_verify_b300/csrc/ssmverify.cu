// libssmverify: CUDA kernels (sm_103a) and the C ABI for the Mamba-layer
// verify / commit / step of speculative decoding.
//
// Method: "The Mamba in the Llama: Distilling and Accelerating Hybrid Models"
// (abstract: hardware-aware speculative decoding for Mamba and hybrid models)
// and the news summary "Llama 3+Mamba强强联手！蒸馏到RNN，推理速度提升1.6倍",
// speculative-decoding section: the Mamba layers run the K draft tokens one
// after another from the cached state, keep no intermediate states, and on
// the first rejected token roll the state back to the last accepted one.
// The recurrence, per (sequence b, head h, token t), with g = h / (H / G):
//   Abar_t = exp(dt_t A_h);  h_t = Abar_t h_{t-1} + (dt_t x_t) B_t^T;
//   y_t = C_t h_t + D_h x_t
// (the discrete-time linear RNN that the method overview derives from the
// continuous-time SSM; C, B, x take the roles of Q, K, V).
//
// Kernel design (B300, HBM-bound on the fp32 state):
//  * One CTA owns a tile of `kRows` head-dim rows p of one (b, h) state slice
//    [P][N] and holds it in registers for all K tokens: 8 rows x 8 state
//    columns per thread, loaded once with 128-bit loads and written back once.
//  * A row group of N/8 lanes spans one row set; lane l holds columns
//    4l..4l+3 and N/2+4l..N/2+4l+3, so one 128-bit warp access covers whole
//    contiguous 256-byte spans (no partial sectors).
//  * Per-token inputs (u = dt x, D x, B, C, Abar) are staged in shared memory
//    in chunks of kTokChunk tokens; B/C rows are broadcast to the row groups.
//  * The update uses paired fp32 instructions (fma.rn.f32x2 / mul.rn.f32x2):
//    h <- Abar * h + (u_p * B_n), two IEEE roundings per element, identical in
//    every kernel so that fused, commit-only and single-step paths agree bit
//    for bit.
//  * y_t[p] = sum_n C_t[n] h_t[p][n]: per-thread partial sums over its 8
//    columns, then a transposing butterfly over the N/8 lanes of the row group
//    (each level halves the rows a lane holds), then D x is added.
//  * The committed state h_j is stored straight from registers right after
//    token j-1 (streaming stores) while the remaining tokens are still
//    computed; j = 0 writes nothing (rollback = no traffic).
//  * Grid: one CTA per (b, h, row tile), row tile fastest, so consecutive
//    CTAs stream consecutive state memory and heads of one B/C group are
//    neighbours (their B/C reads hit L2).

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <stdint.h>

#include "ssmverify.h"

namespace {

constexpr int kTokChunk = 16;  // draft tokens staged in shared memory at a time

enum Mode : int { kVerify = 0, kVerifyCommit = 1, kCommit = 2 };

// Per-N geometry: N/8 lanes per row group, 8 rows per thread.
template <int N>
struct Geo {
    static constexpr int kLanesPerGroup = N / 8;
    static constexpr int kGroupsPerWarp = 32 / kLanesPerGroup;
    static constexpr int kRowsPerWarp = kGroupsPerWarp * 8;
    static constexpr int kRows = kRowsPerWarp > 64 ? kRowsPerWarp : 64;  // rows per CTA
    static constexpr int kWarps = kRows / kRowsPerWarp;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kMinBlocks = 512 / kThreads;  // 128 registers per thread at most
    static_assert(N >= 16 && N <= 256 && (N & (N - 1)) == 0, "dstate must be a power of two in [16, 256]");
};

struct Args {
    const float *state_in;  // read-only state (verify)
    float *state;           // in/out state (commit, verify_commit)
    const void *x, *B, *C, *dt;
    const float *A, *D;
    const int32_t *accept_len;  // nullptr: every token accepted (plain decode)
    float *y;
    uint32_t *dev_status;
    int H, P, G, K, ptiles;
};

__device__ __forceinline__ float load_in(const float *p, int64_t i) { return __ldg(p + i); }
__device__ __forceinline__ float load_in(const __nv_bfloat16 *p, int64_t i) { return __bfloat162float(__ldg(p + i)); }

// Discretisation, shared by every kernel (same calls, same rounding).
__device__ __forceinline__ float ssm_decay(float dt, float A) { return expf(__fmul_rn(dt, A)); }
__device__ __forceinline__ float ssm_input_scale(float dt, float x) { return __fmul_rn(dt, x); }

// One state update of two adjacent columns: h <- Abar h + (u B), two roundings.
__device__ __forceinline__ float2 ssm_update2(float2 h, float2 abar2, float2 u2, float2 b2) {
    return __ffma2_rn(abar2, h, __fmul2_rn(u2, b2));
}

// Keep half of v[0..M) chosen by `bit`, send the other half to the partner
// lane `lane ^ off`, add what the partner sends: afterwards v[0..M/2) holds
// the pair's sums for rows base + (bit ? M/2 : 0) + i.
template <int M>
__device__ __forceinline__ void halve(float *v, bool bit, int off) {
#pragma unroll
    for (int i = 0; i < M / 2; ++i) {
        const float lo = v[i], hi = v[i + M / 2];
        const float keep = bit ? hi : lo;
        const float send = bit ? lo : hi;
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
}

// Reduce 8 per-thread row partials over the LG lanes of a row group.
// Returns in v[0..M) the full sums of local rows `base .. base+M-1` of the
// thread's 8 rows, with M = max(8 / LG, 1); lanes l >= 8 of the group hold
// duplicates.
template <int LG>
__device__ __forceinline__ int reduce_rows(float (&v)[8], int l) {
    int base = 0;
    if constexpr (LG >= 2) { const bool b = l & 1; halve<8>(v, b, 1); base += b ? 4 : 0; }
    if constexpr (LG >= 4) { const bool b = l & 2; halve<4>(v, b, 2); base += b ? 2 : 0; }
    if constexpr (LG >= 8) { const bool b = l & 4; halve<2>(v, b, 4); base += b ? 1 : 0; }
    if constexpr (LG >= 16) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 8);
    if constexpr (LG >= 32) v[0] += __shfl_xor_sync(0xffffffffu, v[0], 16);
    return base;
}

template <typename Tin, int N, int MODE>
__global__ void __launch_bounds__(Geo<N>::kThreads, Geo<N>::kMinBlocks) ssm_scan_kernel(const Args a) {
    using G = Geo<N>;
    constexpr int LG = G::kLanesPerGroup;
    constexpr int ROWS = G::kRows;
    constexpr int THREADS = G::kThreads;
    constexpr bool kWantY = MODE != kCommit;
    constexpr bool kWrite = MODE != kVerify;
    constexpr int M = LG >= 8 ? 1 : 8 / LG;

    __shared__ __align__(16) float sB[kTokChunk][N];
    __shared__ __align__(16) float sC[kWantY ? kTokChunk : 1][kWantY ? N : 4];
    __shared__ __align__(16) float sU[kTokChunk][ROWS];
    __shared__ __align__(16) float sDx[kWantY ? kTokChunk : 1][kWantY ? ROWS : 4];
    __shared__ float sAbar[kTokChunk];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int l = lane % LG;                                        // lane within the row group
    const int rloc = (warp * G::kGroupsPerWarp + lane / LG) * 8;    // first local row of the thread

    int64_t blk = blockIdx.x;
    const int ptile = (int)(blk % a.ptiles);
    blk /= a.ptiles;
    const int h = (int)(blk % a.H);
    const int64_t b = blk / a.H;
    const int g = h / (a.H / a.G);
    const int row0 = ptile * ROWS;
    const int K = a.K;
    const int P = a.P;

    // Accepted prefix j: which state gets committed.
    int jw = K;  // state written after token jw-1; 0 = no write
    if (kWrite && a.accept_len != nullptr) {
        const int j = __ldg(a.accept_len + b);
        if (j < 0 || j > K) {
            if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_BAD_ACCEPT_LEN);
            jw = 0;
        } else {
            jw = j;
        }
    }
    if (MODE == kCommit && jw == 0) return;  // rollback to the cached state: nothing to do
    const int T = (MODE == kCommit) ? jw : K;

    // Load this thread's 8 rows x 8 columns of the cached state h_0.
    const int c0 = 4 * l, c1 = N / 2 + 4 * l;
    const int64_t sbase = (b * a.H + h) * (int64_t)P * N;
    const float *sin = (MODE == kVerify) ? a.state_in : a.state;
    float2 hs[8][4];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int p = row0 + rloc + r;
        float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
        if (p < P) {
            const float *row = sin + sbase + (int64_t)p * N;
            if (MODE == kVerify) {
                v0 = __ldg(reinterpret_cast<const float4 *>(row + c0));
                v1 = __ldg(reinterpret_cast<const float4 *>(row + c1));
            } else {
                v0 = __ldcs(reinterpret_cast<const float4 *>(row + c0));
                v1 = __ldcs(reinterpret_cast<const float4 *>(row + c1));
            }
        }
        hs[r][0] = make_float2(v0.x, v0.y);
        hs[r][1] = make_float2(v0.z, v0.w);
        hs[r][2] = make_float2(v1.x, v1.y);
        hs[r][3] = make_float2(v1.z, v1.w);
    }

    const Tin *xp = static_cast<const Tin *>(a.x);
    const Tin *Bp = static_cast<const Tin *>(a.B);
    const Tin *Cp = static_cast<const Tin *>(a.C);
    const Tin *dtp = static_cast<const Tin *>(a.dt);
    const float Ah = __ldg(a.A + h);
    const float Dh = kWantY ? __ldg(a.D + h) : 0.f;

    for (int t0 = 0; t0 < T; t0 += kTokChunk) {
        const int tc = min(kTokChunk, T - t0);
        if (t0 > 0) __syncthreads();  // the previous chunk's readers are done

        // Stage the chunk's inputs: Abar, u = dt x, D x, B, C.
        for (int i = tid; i < tc; i += THREADS) {
            const float dtv = load_in(dtp, ((b * K + t0 + i) * a.H + h));
            sAbar[i] = ssm_decay(dtv, Ah);
        }
        for (int i = tid; i < tc * ROWS; i += THREADS) {
            const int t = i / ROWS, r = i % ROWS, p = row0 + r;
            const int64_t bt = b * K + t0 + t;
            const float dtv = load_in(dtp, bt * a.H + h);
            const float xv = p < P ? load_in(xp, (bt * a.H + h) * P + p) : 0.f;
            sU[t][r] = ssm_input_scale(dtv, xv);
            if (kWantY) sDx[t][r] = __fmul_rn(Dh, xv);
        }
        for (int i = tid; i < tc * N; i += THREADS) {
            const int t = i / N, n = i % N;
            const int64_t off = ((b * K + t0 + t) * a.G + g) * N + n;
            sB[t][n] = load_in(Bp, off);
            if (kWantY) sC[t][n] = load_in(Cp, off);
        }
        __syncthreads();

        for (int t = 0; t < tc; ++t) {
            // h_t = Abar_t h_{t-1} + u_t B_t^T for the thread's 64 elements.
            const float abar = sAbar[t];
            const float2 ab2 = make_float2(abar, abar);
            const float4 b0 = *reinterpret_cast<const float4 *>(&sB[t][c0]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&sB[t][c1]);
            const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                                  make_float2(b1.z, b1.w)};
            const float4 u0 = *reinterpret_cast<const float4 *>(&sU[t][rloc]);
            const float4 u1 = *reinterpret_cast<const float4 *>(&sU[t][rloc + 4]);
            const float ur[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float2 u2 = make_float2(ur[r], ur[r]);
#pragma unroll
                for (int k = 0; k < 4; ++k) hs[r][k] = ssm_update2(hs[r][k], ab2, u2, bp[k]);
            }

            if constexpr (kWantY) {
                // y_t[p] = sum_n C_t[n] h_t[p][n] + D x_t[p].
                const float4 q0 = *reinterpret_cast<const float4 *>(&sC[t][c0]);
                const float4 q1 = *reinterpret_cast<const float4 *>(&sC[t][c1]);
                const float2 cp[4] = {make_float2(q0.x, q0.y), make_float2(q0.z, q0.w), make_float2(q1.x, q1.y),
                                      make_float2(q1.z, q1.w)};
                float acc[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    float2 s = __fmul2_rn(cp[0], hs[r][0]);
                    s = __ffma2_rn(cp[1], hs[r][1], s);
                    s = __ffma2_rn(cp[2], hs[r][2], s);
                    s = __ffma2_rn(cp[3], hs[r][3], s);
                    acc[r] = s.x + s.y;
                }
                const int base = reduce_rows<LG>(acc, l);
                if (l < 8) {
                    const int64_t ybase = ((b * K + t0 + t) * a.H + h) * P;
#pragma unroll
                    for (int i = 0; i < M; ++i) {
                        const int rl = rloc + base + i;
                        const int p = row0 + rl;
                        if (p < P) __stcs(a.y + ybase + p, acc[i] + sDx[t][rl]);
                    }
                }
            }

            if (kWrite && t0 + t + 1 == jw) {
                // Commit h_j in place, straight from registers.
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int p = row0 + rloc + r;
                    if (p < P) {
                        float *row = a.state + sbase + (int64_t)p * N;
                        __stcs(reinterpret_cast<float4 *>(row + c0),
                               make_float4(hs[r][0].x, hs[r][0].y, hs[r][1].x, hs[r][1].y));
                        __stcs(reinterpret_cast<float4 *>(row + c1),
                               make_float4(hs[r][2].x, hs[r][2].y, hs[r][3].x, hs[r][3].y));
                    }
                }
            }
        }
    }
}

// ----------------------------------------------------------------------------- host side

thread_local int g_last_cuda_error = 0;

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(const Range &a, const Range &b) { return a.lo < b.hi && b.lo < a.hi; }

Range range_of(const void *p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Sizes {
    int64_t state, x, bc, dt, hd, y, acc;  // bytes
};

int check_desc(const ssm_desc_t *d) {
    if (d == nullptr) return SSM_ERR_NULL;
    if (d->reserved != 0) return SSM_ERR_SHAPE;
    if (d->batch < 0 || d->nheads < 1 || d->headdim < 1 || d->dstate < 1 || d->ngroups < 1 || d->ntok < 1)
        return SSM_ERR_SHAPE;
    if (d->nheads % d->ngroups != 0) return SSM_ERR_SHAPE;
    if (d->in_dtype != SSM_F32 && d->in_dtype != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    switch (d->dstate) {
        case 16: case 32: case 64: case 128: case 256: break;
        default: return SSM_ERR_UNSUPPORTED;
    }
    return SSM_OK;
}

int rows_per_cta(int N) {
    switch (N) {
        case 16: return Geo<16>::kRows;
        case 32: return Geo<32>::kRows;
        case 64: return Geo<64>::kRows;
        case 128: return Geo<128>::kRows;
        default: return Geo<256>::kRows;
    }
}

Sizes sizes_of(const ssm_desc_t *d) {
    const int64_t eb = d->in_dtype == SSM_BF16 ? 2 : 4;
    const int64_t bk = (int64_t)d->batch * d->ntok;
    Sizes s;
    s.state = (int64_t)d->batch * d->nheads * d->headdim * d->dstate * 4;
    s.x = bk * d->nheads * d->headdim * eb;
    s.bc = bk * d->ngroups * d->dstate * eb;
    s.dt = bk * d->nheads * eb;
    s.hd = (int64_t)d->nheads * 4;
    s.y = bk * d->nheads * d->headdim * 4;
    s.acc = (int64_t)d->batch * 4;
    return s;
}

template <typename Tin, int N, int MODE>
cudaError_t launch_t(const Args &a, int64_t nblocks, cudaStream_t s) {
    ssm_scan_kernel<Tin, N, MODE><<<(unsigned)nblocks, Geo<N>::kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(int in_dtype, int N, const Args &a, int64_t nblocks, cudaStream_t s) {
    if (in_dtype == SSM_BF16) {
        switch (N) {
            case 16: return launch_t<__nv_bfloat16, 16, MODE>(a, nblocks, s);
            case 32: return launch_t<__nv_bfloat16, 32, MODE>(a, nblocks, s);
            case 64: return launch_t<__nv_bfloat16, 64, MODE>(a, nblocks, s);
            case 128: return launch_t<__nv_bfloat16, 128, MODE>(a, nblocks, s);
            default: return launch_t<__nv_bfloat16, 256, MODE>(a, nblocks, s);
        }
    }
    switch (N) {
        case 16: return launch_t<float, 16, MODE>(a, nblocks, s);
        case 32: return launch_t<float, 32, MODE>(a, nblocks, s);
        case 64: return launch_t<float, 64, MODE>(a, nblocks, s);
        case 128: return launch_t<float, 128, MODE>(a, nblocks, s);
        default: return launch_t<float, 256, MODE>(a, nblocks, s);
    }
}

// Validate everything on the host, then launch. `written` lists the buffers
// the call writes; every one must be disjoint from every other buffer.
int run(int mode, const ssm_desc_t *d, const float *state_in, float *state, const void *x, const void *B,
        const void *C, const void *dt, const float *A, const float *D, const int32_t *accept_len, float *y,
        uint32_t *dev_status, void *stream) {
    int rc = check_desc(d);
    if (rc != SSM_OK) return rc;
    const int N = d->dstate;
    const int ROWS = rows_per_cta(N);
    const int64_t ptiles = (d->headdim + ROWS - 1) / ROWS;
    const int64_t nblocks = (int64_t)d->batch * d->nheads * ptiles;
    if (nblocks > 0x7fffffffLL) return SSM_ERR_SHAPE;
    if (d->batch == 0) return SSM_OK;

    const bool want_y = mode != kCommit;
    const bool writes_state = mode != kVerify;
    const void *st = writes_state ? static_cast<const void *>(state) : static_cast<const void *>(state_in);
    if (st == nullptr || x == nullptr || B == nullptr || dt == nullptr || A == nullptr) return SSM_ERR_NULL;
    if (want_y && (C == nullptr || D == nullptr || y == nullptr)) return SSM_ERR_NULL;
    if (mode == kCommit && accept_len == nullptr) return SSM_ERR_NULL;

    const uintptr_t eb = d->in_dtype == SSM_BF16 ? 2 : 4;
    if (!aligned(st, 16) || !aligned(x, eb) || !aligned(B, eb) || !aligned(dt, eb) || !aligned(A, 4))
        return SSM_ERR_ALIGN;
    if (want_y && (!aligned(C, eb) || !aligned(D, 4) || !aligned(y, 4))) return SSM_ERR_ALIGN;
    if (accept_len != nullptr && !aligned(accept_len, 4)) return SSM_ERR_ALIGN;
    if (dev_status != nullptr && !aligned(dev_status, 4)) return SSM_ERR_ALIGN;

    // Every buffer of the call with whether the call writes it; a written
    // buffer must be disjoint from every other one.
    const Sizes sz = sizes_of(d);
    Range bufs[10];
    bool written[10];
    int nb = 0;
    auto add = [&](const void *p, int64_t bytes, bool w) {
        bufs[nb] = range_of(p, bytes);
        written[nb++] = w;
    };
    add(st, sz.state, writes_state);
    add(x, sz.x, false);
    add(B, sz.bc, false);
    add(dt, sz.dt, false);
    add(A, sz.hd, false);
    if (want_y) {
        add(C, sz.bc, false);
        add(D, sz.hd, false);
        add(y, sz.y, true);
    }
    if (accept_len != nullptr) add(accept_len, sz.acc, false);
    if (dev_status != nullptr) add(dev_status, 4, true);
    for (int i = 0; i < nb; ++i) {
        if (!written[i]) continue;
        for (int k = 0; k < nb; ++k)
            if (k != i && overlaps(bufs[i], bufs[k])) return SSM_ERR_ALIAS;
    }

    Args a;
    a.state_in = state_in;
    a.state = state;
    a.x = x;
    a.B = B;
    a.C = C;
    a.dt = dt;
    a.A = A;
    a.D = D;
    a.accept_len = accept_len;
    a.y = y;
    a.dev_status = dev_status;
    a.H = d->nheads;
    a.P = d->headdim;
    a.G = d->ngroups;
    a.K = d->ntok;
    a.ptiles = (int)ptiles;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (mode) {
        case kVerify: e = launch_mode<kVerify>(d->in_dtype, N, a, nblocks, s); break;
        case kCommit: e = launch_mode<kCommit>(d->in_dtype, N, a, nblocks, s); break;
        default: e = launch_mode<kVerifyCommit>(d->in_dtype, N, a, nblocks, s); break;
    }
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return SSM_ERR_CUDA;
    }
    return SSM_OK;
}

}  // namespace

extern "C" {

int ssm_verify(const ssm_desc_t *desc, const float *state, const void *x, const void *B, const void *C,
               const void *dt, const float *A, const float *D, float *y, void *stream) {
    return run(kVerify, desc, state, nullptr, x, B, C, dt, A, D, nullptr, y, nullptr, stream);
}

int ssm_commit(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *dt,
               const float *A, const int32_t *accept_len, uint32_t *dev_status, void *stream) {
    return run(kCommit, desc, nullptr, state, x, B, nullptr, dt, A, nullptr, accept_len, nullptr, dev_status,
               stream);
}

int ssm_verify_commit(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *C,
                      const void *dt, const float *A, const float *D, const int32_t *accept_len, float *y,
                      uint32_t *dev_status, void *stream) {
    if (accept_len == nullptr && desc != nullptr && desc->batch > 0) return SSM_ERR_NULL;
    return run(kVerifyCommit, desc, nullptr, state, x, B, C, dt, A, D, accept_len, y, dev_status, stream);
}

int ssm_step(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *C, const void *dt,
             const float *A, const float *D, float *y, void *stream) {
    if (desc != nullptr && desc->ntok != 1) return SSM_ERR_SHAPE;
    return run(kVerifyCommit, desc, nullptr, state, x, B, C, dt, A, D, nullptr, y, nullptr, stream);
}

const char *ssm_strerror(int code) {
    switch (code) {
        case SSM_OK: return "ok";
        case SSM_ERR_NULL: return "a required pointer or the descriptor is NULL";
        case SSM_ERR_SHAPE: return "a dimension is out of range (or nheads % ngroups != 0, or ntok < 1)";
        case SSM_ERR_UNSUPPORTED: return "unsupported dstate (16/32/64/128/256) or input dtype";
        case SSM_ERR_ALIGN: return "a pointer is not aligned as required";
        case SSM_ERR_ALIAS: return "a written buffer overlaps another buffer";
        case SSM_ERR_CUDA: return "the CUDA kernel launch failed (see ssm_last_cuda_error)";
        default: return "unknown error code";
    }
}

int ssm_last_cuda_error(void) { return g_last_cuda_error; }

int ssm_version(void) { return SSM_VERSION; }

}  // extern "C"
