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
// Kernel design (B300, bound by HBM traffic of the fp32 state):
//  * Work unit = a tile of kRows head-dim rows p of one (b, h) state slice
//    [P][N]: kRows * N * 4 contiguous bytes (32 KiB at N = 128).
//  * Persistent grid: (SMs x resident CTAs) CTAs walk the tiles round-robin.
//    While a CTA runs the token loop of one tile, the next tile's state is
//    already streaming into shared memory through a 1-D TMA bulk copy
//    (cp.async.bulk, completion on an mbarrier), so HBM never waits for the
//    arithmetic. Waits on the mbarrier are bounded in time; a CTA that gives
//    up records SSM_STATUS_TIMEOUT, drains its copy (again bounded) and exits.
//  * The tile's state lives in registers for all tokens: 8 rows x 8 columns
//    per thread. A row group of N/8 lanes spans one row set; lane l holds
//    columns 4l..4l+3 and N/2+4l..N/2+4l+3, so every warp-wide 128-bit access
//    covers whole 256-byte spans.
//  * Per-token inputs are staged in shared memory kTC tokens at a time with
//    vector loads issued together: Abar = exp(dt A), u = dt x, D x, B, C.
//  * Update with paired fp32 instructions: h <- Abar * h + (u_p * B_n), two
//    IEEE roundings per element, in one device function shared by every
//    flavour, so fused, commit-only, replay and single-step paths agree bit
//    for bit.
//  * y_t[p] = sum_n C_t[n] h_t[p][n]: per-thread partial sums over its 8
//    columns, then a transposing butterfly over the N/8 lanes of the row group
//    (each level halves the rows a lane holds), then D x is added.
//  * A launch runs up to two phases over each tile: a replay phase that
//    advances the state over an accepted prefix of a replay block (no y), and
//    a verify phase over the K draft tokens (y for every token). The state is
//    written once: after the replay phase, or in the verify phase right after
//    token j-1 (streaming stores straight from registers); j = 0 writes nothing.

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <atomic>
#include <stdint.h>

#include "ssmverify.h"

namespace {

constexpr int kTC = 8;                              // draft tokens staged in shared memory at a time
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // give up on a bulk copy after 1 s
constexpr uint32_t kWaitLimitIters = 1u << 26;      // ... or after this many polls, whichever first

enum Flavour : int {
    kVerify = 0,        // verify phase only; the state is read-only
    kVerifyCommit = 1,  // verify phase; h_j written after token j-1 of the verify block
    kCommit = 2,        // replay phase only (j = accept_len); h_j written; j = 0 tiles skipped
    kCommitVerify = 3,  // replay phase, h_j written, then the verify phase from h_j
};

template <int F>
struct Flav {
    static constexpr bool kReplay = F == kCommit || F == kCommitVerify;
    static constexpr bool kVerifyPhase = F != kCommit;
    static constexpr bool kWriteInVerify = F == kVerifyCommit;
};

// Per-N geometry: N/8 lanes per row group, 8 rows per thread.
template <int N>
struct Geo {
    static constexpr int kLanesPerGroup = N / 8;
    static constexpr int kGroupsPerWarp = 32 / kLanesPerGroup;
    static constexpr int kRowsPerWarp = kGroupsPerWarp * 8;
    static constexpr int kRows = kRowsPerWarp > 64 ? kRowsPerWarp : 64;  // rows per tile
    static constexpr int kWarps = kRows / kRowsPerWarp;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kMinBlocks = 512 / kThreads;  // 128 registers per thread at most
    static_assert(N >= 16 && N <= 256 && (N & (N - 1)) == 0, "dstate must be a power of two in [16, 256]");
};

// Dynamic shared memory layout (byte offsets). The state buffer comes first
// (the bulk copy destination, 128-byte aligned).
template <int N, bool WANT_Y>
struct Smem {
    static constexpr int kRows = Geo<N>::kRows;
    static constexpr int kState = 0;                                    // float [kRows][N]
    static constexpr int kB = kState + kRows * N * 4;                   // float [kTC][N]
    static constexpr int kC = kB + kTC * N * 4;                         // float [kTC][N]     (y only)
    static constexpr int kU = kC + (WANT_Y ? kTC * N * 4 : 0);           // float [kTC][kRows]
    static constexpr int kDx = kU + kTC * kRows * 4;                    // float [kTC][kRows] (y only)
    static constexpr int kAbar = kDx + (WANT_Y ? kTC * kRows * 4 : 0);   // float [kTC]
    static constexpr int kBytes = kAbar + kTC * 4;
};

// One block of draft tokens and its inputs (layouts in ssmverify.h).
struct Block {
    const void *x, *B, *C, *dt;
    int K;        // tokens in the block: the extent of the token dimension
    int vec_x;    // x rows may be read 8 elements at a time with 16-byte loads
    int vec_bc;   // B / C rows likewise
};

struct Args {
    const float *state_in;  // state read by the tile loads
    float *state;           // state written (nullptr for verify)
    Block ver;              // verify block: y for every token
    Block rep;              // replay block: advanced over its accepted prefix
    const float *A, *D;
    const int32_t *accept_len;  // verify_commit: j in the verify block (nullptr = all); commit(_verify): j in rep
    float *y;
    uint32_t *dev_status;
    int H, P, G, ptiles;
    long long ntiles;
};

// ----------------------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses (made
// visible to it by a CTA barrier) before later async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(__cvta_generic_to_global(src)), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with `parity` of `bar` to complete; false after the
// time / poll limit.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1; i < kWaitLimitIters; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 1023u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

// ----------------------------------------------------------------------------- loads

__device__ __forceinline__ float ld1(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld1(const __nv_bfloat16 *p) { return __bfloat162float(__ldg(p)); }

// Eight consecutive input elements as loaded (bf16 stays packed until it is
// widened, to keep register pressure low while the state tile is live).
template <typename Tin>
struct Raw8;
template <>
struct Raw8<float> {
    float4 a, b;
};
template <>
struct Raw8<__nv_bfloat16> {
    uint4 a;
};

// Load elements p[0..8); elements at or past `valid` read as 0 and are not
// touched. `vec`: p is 16-byte aligned and the vector load may be used.
__device__ __forceinline__ void ld8(const float *p, bool vec, int valid, Raw8<float> &r) {
    if (vec && valid >= 8) {
        r.a = __ldg(reinterpret_cast<const float4 *>(p));
        r.b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    } else {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = k < valid ? __ldg(p + k) : 0.f;
        r.a = make_float4(v[0], v[1], v[2], v[3]);
        r.b = make_float4(v[4], v[5], v[6], v[7]);
    }
}

__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, bool vec, int valid, Raw8<__nv_bfloat16> &r) {
    if (vec && valid >= 8) {
        r.a = __ldg(reinterpret_cast<const uint4 *>(p));
    } else {
        const unsigned short *q = reinterpret_cast<const unsigned short *>(p);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < valid) w[k / 2] |= (uint32_t)__ldg(q + k) << (16 * (k & 1));
        r.a = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// bf16 is the upper half of an fp32: widening is a 16-bit shift.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void widen(const Raw8<float> &r, float (&v)[8]) {
    v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
    v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
}

__device__ __forceinline__ void widen(const Raw8<__nv_bfloat16> &r, float (&v)[8]) {
    v[0] = bf16_lo(r.a.x); v[1] = bf16_hi(r.a.x); v[2] = bf16_lo(r.a.y); v[3] = bf16_hi(r.a.y);
    v[4] = bf16_lo(r.a.z); v[5] = bf16_hi(r.a.z); v[6] = bf16_lo(r.a.w); v[7] = bf16_hi(r.a.w);
}

__device__ __forceinline__ void st8(float *s, const float (&v)[8]) {
    reinterpret_cast<float4 *>(s)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(s)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// ----------------------------------------------------------------------------- arithmetic (shared by all flavours)

// Discretisation: the same calls, hence the same rounding, everywhere.
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

// ----------------------------------------------------------------------------- tile context

struct Tile {
    long long b;
    int h, g, row0, rows;  // rows: valid rows of this tile (<= kRows)
    long long sbase;       // element offset of the (b, h) state slice
};

__device__ __forceinline__ Tile decode(const Args &a, long long t, int kRows, int N) {
    Tile T;
    const int ptile = (int)(t % a.ptiles);
    const long long bh = t / a.ptiles;
    T.h = (int)(bh % a.H);
    T.b = bh / a.H;
    T.g = T.h / (a.H / a.G);
    T.row0 = ptile * kRows;
    T.rows = min(kRows, a.P - T.row0);
    T.sbase = (T.b * a.H + T.h) * (long long)a.P * N;
    return T;
}

// Stage tokens [t0, t0 + tc) of `blk` for tile T into shared memory laid out
// as Smem<N, SMEMY>; WANT_Y also stages C and D x (the verify phase).
// Work items: an x item is 8 rows of one token (u = dt x and D x), a B/C item
// 8 columns of one token. When every thread has at most one item of each kind
// (dstate >= 64) all of its loads are issued before the first use.
template <typename Tin, int N, bool SMEMY, bool WANT_Y>
__device__ __forceinline__ void stage_chunk(const Args &a, const Block &blk, const Tile &T, int t0, int tc, float Ah,
                                            float Dh, char *smem) {
    static_assert(SMEMY || !WANT_Y, "y staging needs the y layout");
    using S = Smem<N, SMEMY>;
    constexpr int ROWS = Geo<N>::kRows;
    constexpr int THREADS = Geo<N>::kThreads;
    constexpr int XPT = ROWS / 8;  // x items per token
    constexpr int BPT = N / 8;     // B/C items per token
    float *sB = reinterpret_cast<float *>(smem + S::kB);
    float *sC = reinterpret_cast<float *>(smem + S::kC);
    float *sU = reinterpret_cast<float *>(smem + S::kU);
    float *sDx = reinterpret_cast<float *>(smem + S::kDx);
    float *sAbar = reinterpret_cast<float *>(smem + S::kAbar);
    const Tin *xp = static_cast<const Tin *>(blk.x);
    const Tin *Bp = static_cast<const Tin *>(blk.B);
    const Tin *Cp = static_cast<const Tin *>(blk.C);
    const Tin *dtp = static_cast<const Tin *>(blk.dt);
    const int tid = threadIdx.x;
    const long long bt0 = T.b * blk.K + t0;  // (b, t0) in [batch][K]
    const int nx = tc * XPT, nb = tc * BPT;

    auto x_item_store = [&](int i, float dtv, const Raw8<Tin> &xr) {
        const int t = i / XPT, r8 = i % XPT;
        float xv[8], u[8];
        widen(xr, xv);
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] = ssm_input_scale(dtv, xv[e]);
        st8(sU + t * ROWS + 8 * r8, u);
        if (WANT_Y) {
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[e] = __fmul_rn(Dh, xv[e]);
            st8(sDx + t * ROWS + 8 * r8, xv);
        }
    };
    auto x_item_load = [&](int i, float &dtv, Raw8<Tin> &xr) {
        const int t = i / XPT, r8 = i % XPT;
        const long long row = (bt0 + t) * a.H + T.h;
        dtv = ld1(dtp + row);
        ld8(xp + row * a.P + T.row0 + 8 * r8, blk.vec_x, T.rows - 8 * r8, xr);
    };
    auto bc_off = [&](int i) {
        const int t = i / BPT, n8 = i % BPT;
        return ((bt0 + t) * a.G + T.g) * N + 8 * n8;
    };
    auto bc_store = [&](int i, float *dst, const Raw8<Tin> &r) {
        const int t = i / BPT, n8 = i % BPT;
        float v[8];
        widen(r, v);
        st8(dst + t * N + 8 * n8, v);
    };

    if constexpr (kTC * XPT <= THREADS && kTC * BPT <= THREADS) {
        // One item of each kind per thread: issue every load, then convert.
        const bool hx = tid < nx, hb = tid < nb;
        float dtv = 0.f;
        Raw8<Tin> xr, br, cr;
        if (hx) x_item_load(tid, dtv, xr);
        if (hb) {
            ld8(Bp + bc_off(tid), blk.vec_bc, 8, br);
            if (WANT_Y) ld8(Cp + bc_off(tid), blk.vec_bc, 8, cr);
        }
        if (tid < tc) sAbar[tid] = ssm_decay(ld1(dtp + (bt0 + tid) * a.H + T.h), Ah);
        if (hx) x_item_store(tid, dtv, xr);
        if (hb) {
            bc_store(tid, sB, br);
            if (WANT_Y) bc_store(tid, sC, cr);
        }
    } else {
        if (tid < tc) sAbar[tid] = ssm_decay(ld1(dtp + (bt0 + tid) * a.H + T.h), Ah);
#pragma unroll 1
        for (int i = tid; i < nx; i += THREADS) {
            float dtv;
            Raw8<Tin> xr;
            x_item_load(i, dtv, xr);
            x_item_store(i, dtv, xr);
        }
#pragma unroll 1
        for (int i = tid; i < nb; i += THREADS) {
            Raw8<Tin> br, cr;
            ld8(Bp + bc_off(i), blk.vec_bc, 8, br);
            if (WANT_Y) ld8(Cp + bc_off(i), blk.vec_bc, 8, cr);
            bc_store(i, sB, br);
            if (WANT_Y) bc_store(i, sC, cr);
        }
    }
}

// Store the thread's 8 rows of the state (rows at or past `valid` skipped).
template <int N>
__device__ __forceinline__ void store_state(const float2 (&hs)[8][4], float *rows0, int c0, int c1, int valid) {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        if (r < valid) {
            float *row = rows0 + r * N;
            __stcs(reinterpret_cast<float4 *>(row + c0), make_float4(hs[r][0].x, hs[r][0].y, hs[r][1].x, hs[r][1].y));
            __stcs(reinterpret_cast<float4 *>(row + c1), make_float4(hs[r][2].x, hs[r][2].y, hs[r][3].x, hs[r][3].y));
        }
    }
}

// Run `tc` staged tokens (layout Smem<N, SMEMY>) over the thread's state.
// With WANT_Y, y of token t goes to ytok + t * ystride (rows relative to the
// tile). With WRITE, the state after local token `wt` is stored to `srows`.
template <int N, bool SMEMY, bool WANT_Y, bool WRITE>
__device__ __forceinline__ void run_chunk(float2 (&hs)[8][4], const char *smem, int tc, int l, int rloc, int c0,
                                          int c1, float *ytok, long long ystride, int tile_rows, int wt,
                                          float *srows) {
    static_assert(SMEMY || !WANT_Y, "y needs the y layout");
    using S = Smem<N, SMEMY>;
    constexpr int LG = Geo<N>::kLanesPerGroup;
    constexpr int ROWS = Geo<N>::kRows;
    constexpr int M = LG >= 8 ? 1 : 8 / LG;
    const float *sB = reinterpret_cast<const float *>(smem + S::kB);
    const float *sC = reinterpret_cast<const float *>(smem + S::kC);
    const float *sU = reinterpret_cast<const float *>(smem + S::kU);
    const float *sDx = reinterpret_cast<const float *>(smem + S::kDx);
    const float *sAbar = reinterpret_cast<const float *>(smem + S::kAbar);

    for (int t = 0; t < tc; ++t) {
        // h_t = Abar_t h_{t-1} + u_t B_t^T for the thread's 64 elements.
        const float abar = sAbar[t];
        const float2 ab2 = make_float2(abar, abar);
        const float4 b0 = *reinterpret_cast<const float4 *>(sB + t * N + c0);
        const float4 b1 = *reinterpret_cast<const float4 *>(sB + t * N + c1);
        const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                              make_float2(b1.z, b1.w)};
        const float4 u0 = *reinterpret_cast<const float4 *>(sU + t * ROWS + rloc);
        const float4 u1 = *reinterpret_cast<const float4 *>(sU + t * ROWS + rloc + 4);
        const float ur[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float2 u2 = make_float2(ur[r], ur[r]);
#pragma unroll
            for (int k = 0; k < 4; ++k) hs[r][k] = ssm_update2(hs[r][k], ab2, u2, bp[k]);
        }

        if constexpr (WANT_Y) {
            // y_t[p] = sum_n C_t[n] h_t[p][n] + D x_t[p].
            const float4 q0 = *reinterpret_cast<const float4 *>(sC + t * N + c0);
            const float4 q1 = *reinterpret_cast<const float4 *>(sC + t * N + c1);
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
                float *yt = ytok + t * ystride;
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    const int rl = rloc + base + i;
                    if (rl < tile_rows) __stcs(yt + rl, acc[i] + sDx[t * ROWS + rl]);
                }
            }
        }

        if (WRITE && t == wt) store_state<N>(hs, srows, c0, c1, tile_rows - rloc);
    }
}

// Is there work for tile t? Only commit-only launches skip tiles (j = 0 or
// an invalid j: nothing to replay, nothing to write).
template <int F>
__device__ __forceinline__ long long next_work(const Args &a, long long t) {
    if constexpr (F == kCommit) {
        const long long per_b = (long long)a.H * a.ptiles;
        for (; t < a.ntiles; t += gridDim.x) {
            const int j = __ldg(a.accept_len + t / per_b);
            if (j > 0 && j <= a.rep.K) return t;
            if (j != 0 && threadIdx.x == 0 && a.dev_status != nullptr)
                atomicOr(a.dev_status, SSM_STATUS_BAD_ACCEPT_LEN);
        }
        return a.ntiles;
    } else {
        return t;
    }
}

// Register budget: 128 per thread (4 resident 128-thread CTAs at N = 128),
// except commit_verify, whose two phases keep more addresses live next to the
// state tile: 168 per thread (3 CTAs).
template <int N, int F>
constexpr int min_blocks() {
    return F == kCommitVerify ? (65536 / 168 / Geo<N>::kThreads > 0 ? 65536 / 168 / Geo<N>::kThreads : 1)
                              : Geo<N>::kMinBlocks;
}

template <typename Tin, int N, int F>
__global__ void __launch_bounds__(Geo<N>::kThreads, (min_blocks<N, F>())) ssm_tile_kernel(const Args a) {
    using G = Geo<N>;
    using FL = Flav<F>;
    constexpr int LG = G::kLanesPerGroup;
    constexpr int ROWS = G::kRows;
    constexpr bool WANT_Y = FL::kVerifyPhase;
    using S = Smem<N, WANT_Y>;

    extern __shared__ __align__(128) char smem[];
    __shared__ uint64_t bar;
    float *sS = reinterpret_cast<float *>(smem + S::kState);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int l = lane % LG;                                        // lane within the row group
    const int rloc = (warp * G::kGroupsPerWarp + lane / LG) * 8;    // first local row of the thread
    const int c0 = 4 * l, c1 = N / 2 + 4 * l;

    long long t = next_work<F>(a, blockIdx.x);
    if (t >= a.ntiles) return;  // uniform over the CTA

    auto prefetch = [&](long long tt) {
        const Tile T = decode(a, tt, ROWS, N);
        const uint32_t bytes = (uint32_t)T.rows * N * 4;
        mbar_arrive_expect_tx(&bar, bytes);
        bulk_load(sS, a.state_in + T.sbase + (long long)T.row0 * N, bytes, &bar);
    };

    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch(t);
    }
    __syncthreads();

    const float *Aall = a.A;
    uint32_t parity = 0;
    while (t < a.ntiles) {
        const Tile T = decode(a, t, ROWS, N);
        const float Ah = __ldg(Aall + T.h);
        const float Dh = WANT_Y ? __ldg(a.D + T.h) : 0.f;

        // The tile's state: shared memory (filled by the bulk copy) -> registers.
        const bool ok = mbar_wait_bounded(&bar, parity);
        float2 hs[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const float *row = sS + (rloc + r) * N;
            float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
            if (rloc + r < T.rows) {
                v0 = *reinterpret_cast<const float4 *>(row + c0);
                v1 = *reinterpret_cast<const float4 *>(row + c1);
            }
            hs[r][0] = make_float2(v0.x, v0.y);
            hs[r][1] = make_float2(v0.z, v0.w);
            hs[r][2] = make_float2(v1.x, v1.y);
            hs[r][3] = make_float2(v1.z, v1.w);
        }
        const long long tn = next_work<F>(a, t + gridDim.x);
        // Every thread is done with the state buffer and with the previous
        // tile's staged inputs; the vote makes a timeout a CTA-wide decision.
        if (__syncthreads_or(!ok)) {
            if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_TIMEOUT);
            mbar_wait_bounded(&bar, parity);  // drain the copy still in flight, bounded
            return;
        }
        if (tid == 0 && tn < a.ntiles) {
            fence_proxy_async_smem();
            prefetch(tn);
        }
        parity ^= 1u;

        float *srows = (a.state != nullptr) ? a.state + T.sbase + (long long)(T.row0 + rloc) * N : nullptr;

        // Accepted prefix j of this tile's sequence.
        int jr = 0;  // tokens replayed from the replay block
        int jw = -1; // verify-phase token after which the state is written (-1: none)
        if constexpr (FL::kReplay || FL::kWriteInVerify) {
            const int kref = FL::kReplay ? a.rep.K : a.ver.K;
            int j = kref;
            if (a.accept_len != nullptr) {
                j = __ldg(a.accept_len + T.b);
                if (j < 0 || j > kref) {
                    if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_BAD_ACCEPT_LEN);
                    j = 0;
                }
            }
            if (FL::kReplay) jr = j;
            else jw = j - 1;
        }

        if constexpr (FL::kReplay) {
            // Replay phase: advance over tokens 0 .. jr-1 of the replay block, then commit h_jr.
            for (int t0 = 0; t0 < jr; t0 += kTC) {
                const int tc = min(kTC, jr - t0);
                if (t0 > 0) __syncthreads();
                stage_chunk<Tin, N, WANT_Y, false>(a, a.rep, T, t0, tc, Ah, 0.f, smem);
                __syncthreads();
                run_chunk<N, WANT_Y, false, false>(hs, smem, tc, l, rloc, c0, c1, nullptr, 0, T.rows, -1, nullptr);
            }
            if (jr > 0) store_state<N>(hs, srows, c0, c1, T.rows - rloc);
            if (FL::kVerifyPhase && jr > 0) __syncthreads();  // the verify phase restages the buffers
        }

        if constexpr (FL::kVerifyPhase) {
            const int K = a.ver.K;
            float *ytile = a.y + (T.b * K * a.H + T.h) * (long long)a.P + T.row0;
            const long long ystride = (long long)a.H * a.P;
            for (int t0 = 0; t0 < K; t0 += kTC) {
                const int tc = min(kTC, K - t0);
                if (t0 > 0) __syncthreads();
                stage_chunk<Tin, N, true, true>(a, a.ver, T, t0, tc, Ah, Dh, smem);
                __syncthreads();
                run_chunk<N, true, true, FL::kWriteInVerify>(hs, smem, tc, l, rloc, c0, c1, ytile + t0 * ystride,
                                                       ystride, T.rows, jw - t0, srows);
            }
        }
        t = tn;
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

int rows_per_tile(int N) {
    switch (N) {
        case 16: return Geo<16>::kRows;
        case 32: return Geo<32>::kRows;
        case 64: return Geo<64>::kRows;
        case 128: return Geo<128>::kRows;
        default: return Geo<256>::kRows;
    }
}

// Resident CTAs per SM and the SM count, per device (immutable device
// properties, computed once per (kernel, device) and cached).
constexpr int kMaxDevices = 64;

template <typename Tin, int N, int F>
cudaError_t launch_t(const Args &a, cudaStream_t s) {
    constexpr int THREADS = Geo<N>::kThreads;
    constexpr int SMEM = Smem<N, Flav<F>::kVerifyPhase>::kBytes;
    static std::atomic<int> grid_cache[kMaxDevices];  // SMs x resident CTAs, 0 = unknown
    auto kern = ssm_tile_kernel<Tin, N, F>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int full = (dev >= 0 && dev < kMaxDevices) ? grid_cache[dev].load(std::memory_order_relaxed) : 0;
    if (full == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, THREADS, SMEM);
        if (e != cudaSuccess) return e;
        full = sms * (per_sm > 0 ? per_sm : 1);
        if (dev >= 0 && dev < kMaxDevices) grid_cache[dev].store(full, std::memory_order_relaxed);
    }
    const long long grid = a.ntiles < full ? a.ntiles : full;
    kern<<<(unsigned)grid, THREADS, SMEM, s>>>(a);
    return cudaGetLastError();
}

template <int F>
cudaError_t launch_flavour(int in_dtype, int N, const Args &a, cudaStream_t s) {
    if (in_dtype == SSM_BF16) {
        switch (N) {
            case 16: return launch_t<__nv_bfloat16, 16, F>(a, s);
            case 32: return launch_t<__nv_bfloat16, 32, F>(a, s);
            case 64: return launch_t<__nv_bfloat16, 64, F>(a, s);
            case 128: return launch_t<__nv_bfloat16, 128, F>(a, s);
            default: return launch_t<__nv_bfloat16, 256, F>(a, s);
        }
    }
    switch (N) {
        case 16: return launch_t<float, 16, F>(a, s);
        case 32: return launch_t<float, 32, F>(a, s);
        case 64: return launch_t<float, 64, F>(a, s);
        case 128: return launch_t<float, 128, F>(a, s);
        default: return launch_t<float, 256, F>(a, s);
    }
}

// The buffers of one call, and which of them it writes.
struct BufList {
    Range r[16];
    bool w[16];
    int n = 0;
    void add(const void *p, int64_t bytes, bool written) {
        r[n] = range_of(p, bytes);
        w[n++] = written;
    }
    bool disjoint_writes() const {
        for (int i = 0; i < n; ++i) {
            if (!w[i]) continue;
            for (int k = 0; k < n; ++k)
                if (k != i && overlaps(r[i], r[k])) return false;
        }
        return true;
    }
};

struct Call {
    int flavour;
    const float *state_in;  // verify
    float *state;           // every other flavour
    const void *x, *B, *C, *dt;               // verify block
    int rep_ntok;                             // commit_verify: tokens of the replay block
    const void *xr, *Br, *dtr;                // replay block (commit: the call's own x / B / dt)
    const float *A, *D;
    const int32_t *accept_len;
    float *y;
    uint32_t *dev_status;
};

// Validate everything on the host, then launch.
int run(const ssm_desc_t *d, const Call &c, void *stream) {
    int rc = check_desc(d);
    if (rc != SSM_OK) return rc;
    const int F = c.flavour;
    const bool verify_phase = F != kCommit;
    const bool replay = F == kCommit || F == kCommitVerify;
    const int rep_K = F == kCommit ? d->ntok : c.rep_ntok;
    if (F == kCommitVerify && rep_K < 1) return SSM_ERR_SHAPE;
    const int N = d->dstate;
    const int ROWS = rows_per_tile(N);
    const int64_t ptiles = (d->headdim + ROWS - 1) / ROWS;
    const int64_t ntiles = (int64_t)d->batch * d->nheads * ptiles;
    if (d->batch == 0) return SSM_OK;

    const void *st = F == kVerify ? static_cast<const void *>(c.state_in) : static_cast<const void *>(c.state);
    if (st == nullptr || c.A == nullptr) return SSM_ERR_NULL;
    if (verify_phase && (c.x == nullptr || c.B == nullptr || c.C == nullptr || c.dt == nullptr || c.D == nullptr ||
                         c.y == nullptr))
        return SSM_ERR_NULL;
    if (replay && (c.xr == nullptr || c.Br == nullptr || c.dtr == nullptr || c.accept_len == nullptr))
        return SSM_ERR_NULL;

    const uintptr_t eb = d->in_dtype == SSM_BF16 ? 2 : 4;
    if (!aligned(st, 16) || !aligned(c.A, 4)) return SSM_ERR_ALIGN;
    if (verify_phase && (!aligned(c.x, eb) || !aligned(c.B, eb) || !aligned(c.C, eb) || !aligned(c.dt, eb) ||
                         !aligned(c.D, 4) || !aligned(c.y, 4)))
        return SSM_ERR_ALIGN;
    if (replay && (!aligned(c.xr, eb) || !aligned(c.Br, eb) || !aligned(c.dtr, eb))) return SSM_ERR_ALIGN;
    if (c.accept_len != nullptr && !aligned(c.accept_len, 4)) return SSM_ERR_ALIGN;
    if (c.dev_status != nullptr && !aligned(c.dev_status, 4)) return SSM_ERR_ALIGN;

    const int64_t B_ = d->batch, H = d->nheads, P = d->headdim, G = d->ngroups;
    const int64_t state_bytes = B_ * H * P * N * 4;
    BufList bl;
    bl.add(st, state_bytes, F != kVerify);
    bl.add(c.A, H * 4, false);
    if (verify_phase) {
        const int64_t bk = B_ * d->ntok;
        bl.add(c.x, bk * H * P * eb, false);
        bl.add(c.B, bk * G * N * eb, false);
        bl.add(c.C, bk * G * N * eb, false);
        bl.add(c.dt, bk * H * eb, false);
        bl.add(c.D, H * 4, false);
        bl.add(c.y, bk * H * P * 4, true);
    }
    if (replay && F == kCommitVerify) {  // commit's replay block is the call's x / B / dt, listed below
        const int64_t bk = B_ * rep_K;
        bl.add(c.xr, bk * H * P * eb, false);
        bl.add(c.Br, bk * G * N * eb, false);
        bl.add(c.dtr, bk * H * eb, false);
    } else if (F == kCommit) {
        const int64_t bk = B_ * rep_K;
        bl.add(c.xr, bk * H * P * eb, false);
        bl.add(c.Br, bk * G * N * eb, false);
        bl.add(c.dtr, bk * H * eb, false);
    }
    if (c.accept_len != nullptr) bl.add(c.accept_len, B_ * 4, false);
    if (c.dev_status != nullptr) bl.add(c.dev_status, 4, true);
    if (!bl.disjoint_writes()) return SSM_ERR_ALIAS;

    Args a;
    a.state_in = static_cast<const float *>(st);
    a.state = F == kVerify ? nullptr : c.state;
    const uintptr_t rowb = (uintptr_t)P * eb;
    a.ver.x = c.x;
    a.ver.B = c.B;
    a.ver.C = c.C;
    a.ver.dt = c.dt;
    a.ver.K = d->ntok;
    a.ver.vec_x = verify_phase && aligned(c.x, 16) && rowb % 16 == 0;
    a.ver.vec_bc = verify_phase && aligned(c.B, 16) && aligned(c.C, 16);
    a.rep.x = c.xr;
    a.rep.B = c.Br;
    a.rep.C = nullptr;
    a.rep.dt = c.dtr;
    a.rep.K = rep_K;
    a.rep.vec_x = replay && aligned(c.xr, 16) && rowb % 16 == 0;
    a.rep.vec_bc = replay && aligned(c.Br, 16);
    a.A = c.A;
    a.D = c.D;
    a.accept_len = c.accept_len;
    a.y = c.y;
    a.dev_status = c.dev_status;
    a.H = d->nheads;
    a.P = d->headdim;
    a.G = d->ngroups;
    a.ptiles = (int)ptiles;
    a.ntiles = ntiles;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (F) {
        case kVerify: e = launch_flavour<kVerify>(d->in_dtype, N, a, s); break;
        case kCommit: e = launch_flavour<kCommit>(d->in_dtype, N, a, s); break;
        case kCommitVerify: e = launch_flavour<kCommitVerify>(d->in_dtype, N, a, s); break;
        default: e = launch_flavour<kVerifyCommit>(d->in_dtype, N, a, s); break;
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
               const void *dt, const float *A, const float *D, float *y, uint32_t *dev_status, void *stream) {
    Call c{};
    c.flavour = kVerify;
    c.state_in = state;
    c.x = x; c.B = B; c.C = C; c.dt = dt;
    c.A = A; c.D = D; c.y = y;
    c.dev_status = dev_status;
    return run(desc, c, stream);
}

int ssm_commit(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *dt,
               const float *A, const int32_t *accept_len, uint32_t *dev_status, void *stream) {
    Call c{};
    c.flavour = kCommit;
    c.state = state;
    c.xr = x; c.Br = B; c.dtr = dt;
    c.A = A;
    c.accept_len = accept_len;
    c.dev_status = dev_status;
    return run(desc, c, stream);
}

int ssm_verify_commit(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *C,
                      const void *dt, const float *A, const float *D, const int32_t *accept_len, float *y,
                      uint32_t *dev_status, void *stream) {
    if (accept_len == nullptr && desc != nullptr && desc->batch > 0) return SSM_ERR_NULL;
    Call c{};
    c.flavour = kVerifyCommit;
    c.state = state;
    c.x = x; c.B = B; c.C = C; c.dt = dt;
    c.A = A; c.D = D; c.y = y;
    c.accept_len = accept_len;
    c.dev_status = dev_status;
    return run(desc, c, stream);
}

int ssm_commit_verify(const ssm_desc_t *desc, float *state, int32_t prev_ntok, const void *x_prev,
                      const void *B_prev, const void *dt_prev, const int32_t *accept_len_prev, const void *x,
                      const void *B, const void *C, const void *dt, const float *A, const float *D, float *y,
                      uint32_t *dev_status, void *stream) {
    Call c{};
    c.flavour = kCommitVerify;
    c.state = state;
    c.rep_ntok = prev_ntok;
    c.xr = x_prev; c.Br = B_prev; c.dtr = dt_prev;
    c.accept_len = accept_len_prev;
    c.x = x; c.B = B; c.C = C; c.dt = dt;
    c.A = A; c.D = D; c.y = y;
    c.dev_status = dev_status;
    return run(desc, c, stream);
}

int ssm_step(const ssm_desc_t *desc, float *state, const void *x, const void *B, const void *C, const void *dt,
             const float *A, const float *D, float *y, uint32_t *dev_status, void *stream) {
    if (desc != nullptr && desc->ntok != 1) return SSM_ERR_SHAPE;
    Call c{};
    c.flavour = kVerifyCommit;
    c.state = state;
    c.x = x; c.B = B; c.C = C; c.dt = dt;
    c.A = A; c.D = D; c.y = y;
    c.dev_status = dev_status;
    return run(desc, c, stream);
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
