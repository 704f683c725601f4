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
//  * Work unit = a tile of kRows head-dim rows of one (b, h) state slice
//    [P][N] (64 rows x N, or 32 rows at N = 256): contiguous bytes.
//  * Persistent grid: (SMs x resident CTAs) CTAs walk the tiles round-robin.
//    While a CTA works on one tile, the next tile's state and the raw x / B /
//    C rows of its first kTC draft tokens stream into shared memory through
//    1-D TMA bulk copies completing on one mbarrier, so HBM never waits for
//    the arithmetic. Waits on the mbarrier are bounded in time; a CTA that
//    gives up records SSM_STATUS_TIMEOUT, drains its copies and exits.
//  * y from the attention-like (dual) form of the recurrence over a chunk of
//    up to kTC tokens that starts from state h:
//        y_t = w_t (C_t . h) + sum_{s<=t} L[t,s] (C_t . B_s) u_s + D x_t
//        w_t = exp(A cs_t), L[t,s] = exp(A (cs_t - cs_s)), cs_t = sum_{r<=t} dt_r
//    (C, B, x in the roles of Q, K, V: the correspondence the distillation
//    starts from). h . C^T and C . B^T are dense contractions and run on the
//    tensor cores (mma.sync m16n8k8 tf32, fp32 accumulation), with the
//    fp32 operands split into a tf32 high part and a tf32 low part so that
//    the products keep fp32 accuracy; bf16 inputs are exact in tf32 and need
//    no split. The state stays in registers in the mma fragment layout: warp
//    w owns 16 rows of the tile, a thread rows g and g + 8 and, of each 8
//    columns, those the fragment gives it.
//  * The state advances only as far as needed: up to the committed token j
//    (and through the chunk when more chunks follow); verify-only launches
//    do not advance it at all for K <= kTC. At N <= 128 the advance over the
//    first m tokens of a chunk is the recurrence regrouped into one rank-8
//    tensor-core product,
//        h <- lambda h + sum_{s<m} w_s u_s B_s^T,  lambda = prod_{s<m} Abar_s,
//        w_s = prod_{s<r<m} Abar_r,
//    formed from zero and added to lambda h by one fp32 fma per element
//    (round to nearest), with the register state as the mma D fragment. The
//    committed state is always formed by that same arithmetic over the same
//    tokens, so the fused, commit-only and deferred-commit paths, and a
//    block that ends at the committed token, write it bit for bit alike. At
//    N = 256 (two warps per band) the state takes the exact recurrence
//    h <- Abar h + u B token by token (paired fp32 instructions).
//  * Flavours: a replay phase (advance over the accepted prefix of a replay
//    block, write h_j) and/or a verify phase (y for every draft token; the
//    fused flavour writes h_j, j = accept_len, straight from registers).

#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include <atomic>
#include <stdint.h>

#include "ssmverify.h"
#include "ssm_internal.h"

namespace {

constexpr int kTC = 8;                              // draft tokens per chunk (one mma n-block)
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // give up on a bulk copy after 1 s
constexpr uint32_t kWaitLimitIters = 1u << 26;      // ... or after this many polls, whichever first
constexpr int kThreads = 128;                       // 4 warps per CTA

enum Flavour : int {
    kVerify = 0,        // verify phase only; the state is read-only
    kVerifyCommit = 1,  // verify phase; h_j written after token j-1 of the verify block
    kCommit = 2,        // replay phase only (j = accept_len); h_j written; j = 0 tiles skipped
    kCommitVerify = 3,  // replay phase, h_j written, then the verify phase from h_j
};

// Option bits OR-ed into a flavour: the state is reached through a slot map
// (a pool), and every tile starts from h = 0 without reading a state.
constexpr int kPoolBit = 8;
constexpr int kZeroBit = 16;

template <int F>
struct Flav {
    static constexpr int kBase = F & 7;
    static constexpr bool kReplay = kBase == kCommit || kBase == kCommitVerify;
    static constexpr bool kVerifyPhase = kBase != kCommit;
    static constexpr bool kWriteInVerify = kBase == kVerifyCommit;
    static constexpr bool kPool = (F & kPoolBit) != 0;
    static constexpr bool kZero = (F & kZeroBit) != 0;
};

// Per-N geometry. A band is 16 rows (one mma M block); WPB warps share a
// band by columns (2 at N = 256, else 1). A thread holds rows g and g + 8 of
// its band and NC of the band's columns: the 4-column chunks tq, tq + 4,
// tq + 8, ... (tq = lane % 4) of its warp's column range.
template <int N>
struct Geo {
    static constexpr int kWPB = N > 128 ? N / 128 : 1;   // warps per band
    static constexpr int kNCW = N / kWPB;                // columns per warp
    static constexpr int kNC = kNCW / 4;                 // columns per thread (and per row)
    static constexpr int kKB = kNCW / 8;                 // mma k-blocks per warp
    static constexpr int kBands = 4 / kWPB;
    static constexpr int kRows = 16 * kBands;            // rows per tile
    // Padded row of a thread's slots in the staged B / C (floats). With one
    // warp per band the mma-fragment reads (8-byte loads of lane g*4+tq's row,
    // 4-byte loads of row tq*4 + g/2) hit 32 distinct banks when the row is
    // 2 mod 32 floats long; the token-by-token recurrence (two warps per band)
    // reads 16-byte vectors and needs a multiple of 4.
    static constexpr int kPad = kWPB == 1 ? kNC + 2 : kNC + 4;
    // Row strides (floats) of the staged u = dt x and D x, [kTC][stride]: the
    // loads of u[tq][g] and of D x[2tq + e][g] by the 32 lanes land on
    // distinct banks with 8 and 4 floats of padding.
    static constexpr int kUS = kRows + 8;
    static constexpr int kDS = kRows + 4;
    static_assert(N >= 16 && N <= 256 && (N & (N - 1)) == 0, "dstate must be a power of two in [16, 256]");
};

// Dynamic shared memory layout of one flavour (byte offsets, every region a
// multiple of 16 bytes). The state tile first (bulk copy destination). Two
// raw buffers, used by alternate tiles: the first chunk's x / B / C rows of
// the verify phase (of the replay phase in the commit-only flavour) as stored
// in global memory (bulk-copy destinations), so that the next tile's copies
// can be issued before this tile's rows are converted.
// Staged areas (fp32, what the arithmetic reads): B and C with each thread's
// slots contiguous ([token][warp column half][tq][kPad]), u = dt x and D x
// per row, Abar, cs (cumulative dt) and w per token.
template <typename Tin, int N, int F>
struct Lay {
    using G = Geo<N>;
    static constexpr int ROWS = G::kRows;
    static constexpr bool R = Flav<F>::kReplay;
    static constexpr bool V = Flav<F>::kVerifyPhase;
    // the replay's first chunk travels with the tile's copies only in the commit-only flavour; the
    // deferred-commit flavours stage it from global memory into the verify phase's arrays (below)
    static constexpr bool RR = R && !V;
    static constexpr int E = (int)sizeof(Tin);
    static constexpr int BC = kTC * G::kWPB * 4 * G::kPad * 4;        // one permuted B or C chunk
    static constexpr int kState = 0;                                    // float [ROWS][N]
    // one raw buffer (offsets within it)
    static constexpr int oVx = 0;                                       // Tin [kTC][ROWS]
    static constexpr int oVB = oVx + (V ? kTC * ROWS * E : 0);          // Tin [kTC][N]
    static constexpr int oVC = oVB + (V ? kTC * N * E : 0);             // Tin [kTC][N]
    static constexpr int oRx = oVC + (V ? kTC * N * E : 0);             // Tin [kTC][ROWS]
    static constexpr int oRB = oRx + (RR ? kTC * ROWS * E : 0);         // Tin [kTC][N]
    static constexpr int kRawBytes = oRB + (RR ? kTC * N * E : 0);
    static constexpr int kRaw = kState + ROWS * N * 4;                  // 2 raw buffers
    static constexpr int kVB = kRaw + 2 * kRawBytes;                    // float, permuted
    static constexpr int kVC = kVB + (V ? BC : 0);                      // float, permuted
    static constexpr int kVU = kVC + (V ? BC : 0);                      // float [kTC][kUS]
    static constexpr int kVDx = kVU + (V ? kTC * G::kUS * 4 : 0);       // float [kTC][kDS]
    static constexpr int kVAbar = kVDx + (V ? kTC * G::kDS * 4 : 0);    // float [kTC]
    static constexpr int kVCs = kVAbar + (V ? kTC * 4 : 0);             // float [kTC]
    static constexpr int kVW = kVCs + (V ? kTC * 4 : 0);                // float [kTC]
    static constexpr int kXch = kVW + (V ? kTC * 4 : 0);                // float [bands][32][8] (N = 256)
    static constexpr int kXchEnd = kXch + (V && G::kWPB > 1 ? G::kBands * 32 * 8 * 4 : 0);
    // the replay's staged arrays: their own, or with a verify phase the verify phase's, which is
    // staged only once the replay is done
    static constexpr int kRB = V ? kVB : kXchEnd;                       // float, permuted
    static constexpr int kRU = V ? kVU : kRB + (R ? BC : 0);            // float [kTC][kUS]
    static constexpr int kRAbar = V ? kVAbar : kRU + (R ? kTC * G::kUS * 4 : 0);  // float [kTC]
    static constexpr int kBytes = V ? kXchEnd : kRAbar + (R ? kTC * 4 : 0);
    static_assert(kRawBytes % 16 == 0 && kRaw % 128 == 0, "bulk-copy destinations must be 16-byte aligned");
};

// One block of draft tokens and its inputs (layouts in ssmverify.h).
struct Block {
    const void *x, *B, *C, *dt;
    int K;        // tokens in the block: the extent of the token dimension
    int vec_x;    // x rows may be read 8 elements at a time with 16-byte loads
    int vec_bc;   // B / C rows likewise
    int tma;      // the first chunk's x / B / C rows may be bulk-copied (16-byte aligned rows)
};

// Division by a divisor fixed for the launch, as a multiply-high and a shift
// (the round-up method of Granlund and Montgomery, "Division by invariant
// integers using multiplication", 1994): with s = ceil(log2 d) and
// mul = floor(2^32 (2^s - d) / d) + 1, n / d = (mulhi(n, mul) + n) >> s for
// every 32-bit n, the sum taken in 64 bits. Divisors in [1, 2^31].
struct FastDiv {
    uint32_t d, mul, shift;
};
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv &f) {
    return (uint32_t)(((unsigned long long)__umulhi(n, f.mul) + n) >> f.shift);
}
inline FastDiv make_fdiv(uint32_t d) {
    FastDiv f{d, 0u, 0u};
    while ((1ull << f.shift) < d) ++f.shift;
    f.mul = (uint32_t)(((1ull << 32) * ((1ull << f.shift) - d)) / d + 1);
    return f;
}

struct Args {
    FastDiv fd_ptiles, fd_H, fd_bpl, fd_hpg;  // tile decode: P-tiles, heads, sequences per layer, heads per group
    const float *state_in;  // state read by the tile loads
    float *state;           // state written (nullptr for verify)
    const int32_t *slot;    // pool flavours: slot of each sequence (nullptr: sequence b uses slot b)
    int nslots;             // pool flavours: slots in the pool
    Block ver;              // verify block: y for every token
    Block rep;              // replay block: advanced over its accepted prefix
    const float *A, *D;
    const int32_t *accept_len;  // verify_commit: j in the verify block (nullptr = all); commit(_verify): j in rep
    float *y;
    uint32_t *dev_status;
    int H, P, G, ptiles;
    int bpl;  // sequences per layer: a layer stack is one batch of nlayers x bpl sequences
    long long ntiles;
};

// The kernels' dynamic shared memory (laid out by Lay).
extern __shared__ __align__(128) char ssm_smem[];

template <typename T>
__device__ __forceinline__ T *sm(int off) { return reinterpret_cast<T *>(ssm_smem + off); }

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

// The same, with the source lines marked first to be evicted from L2 (data read once).
__device__ __forceinline__ void bulk_load_once(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(__cvta_generic_to_global(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
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

// tf32 high part of x (rounded toward zero: the top 19 bits), as the bit
// pattern mma reads. Toward zero is one instruction on sm_103a, where the
// rounding conversion issues about three and a half.
__device__ __forceinline__ uint32_t tf32_hi(float x) {
    uint32_t r;
    asm("cvt.rz.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

// d += a (16x8, row) * b (8x8, col), tf32 operands, fp32 accumulation.
__device__ __forceinline__ void mma_tf32(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ----------------------------------------------------------------------------- loads

__device__ __forceinline__ float ld1(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ld1(const __nv_bfloat16 *p) { return __bfloat162float(__ldg(p)); }

// Eight consecutive input elements as loaded (bf16 stays packed until it is
// widened, to keep register pressure low).
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

// The same eight elements from shared memory (16-byte aligned).
__device__ __forceinline__ void lds8(const float *p, Raw8<float> &r) {
    r.a = reinterpret_cast<const float4 *>(p)[0];
    r.b = reinterpret_cast<const float4 *>(p)[1];
}
__device__ __forceinline__ void lds8(const __nv_bfloat16 *p, Raw8<__nv_bfloat16> &r) {
    r.a = *reinterpret_cast<const uint4 *>(p);
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

__device__ __forceinline__ void st4(float *s, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(s) = make_float4(a, b, c, d);
}

// Four consecutive staged B / C slots: one 16-byte store where the padded
// rows keep 16-byte alignment (Geo::kPad a multiple of 4), else two 8-byte stores.
template <int N>
__device__ __forceinline__ void st_slots(float *s, float a, float b, float c, float d) {
    if constexpr (Geo<N>::kPad % 4 == 0) {
        st4(s, a, b, c, d);
    } else {
        reinterpret_cast<float2 *>(s)[0] = make_float2(a, b);
        reinterpret_cast<float2 *>(s)[1] = make_float2(c, d);
    }
}

// ----------------------------------------------------------------------------- arithmetic (shared by all flavours)

// Discretisation: the same calls, hence the same rounding, everywhere.
__device__ __forceinline__ float ssm_decay(float dt, float A) { return expf(__fmul_rn(dt, A)); }
__device__ __forceinline__ float ssm_input_scale(float dt, float x) { return __fmul_rn(dt, x); }

// One state update of two adjacent slots: h <- Abar h + (u B), two roundings.
__device__ __forceinline__ float2 ssm_update2(float2 h, float2 abar2, float2 u2, float2 b2) {
    return __ffma2_rn(abar2, h, __fmul2_rn(u2, b2));
}

// Staged position of state column n (within [0, N)): the permuted B / C
// arrays keep each thread's slots contiguous. Column n belongs to warp
// column half n / kNCW, to the thread with tq = (n / 4) % 4 of that half, at
// slot 4 * ((n / 4) / 4) + n % 4.
template <int N>
__device__ __forceinline__ int perm_index(int n) {
    using G = Geo<N>;
    const int half = n / G::kNCW, n2 = n % G::kNCW, c = n2 / 4;
    return (half * 4 + (c & 3)) * G::kPad + 4 * (c >> 2) + (n2 & 3);
}

// ----------------------------------------------------------------------------- tile context

struct Tile {
    long long b;           // sequence of the call (layer-major over a layer stack)
    int bs, lay;           // sequence within its layer, layer
    int h, g, row0, rows;  // rows: valid rows of this tile (<= kRows)
    long long sbase;       // element offset of the (b, h) state slice
    bool ok;               // the sequence's pool slot is valid (else nothing is written)
};

template <bool POOL>
__device__ __forceinline__ Tile decode(const Args &a, long long t, int kRows, int N) {
    Tile T;
    const uint32_t tt = (uint32_t)t;  // the host keeps the tile count below 2^31
    const uint32_t bh = fdiv(tt, a.fd_ptiles);
    const int ptile = (int)(tt - bh * (uint32_t)a.ptiles);
    const uint32_t bb = fdiv(bh, a.fd_H);
    T.h = (int)(bh - bb * (uint32_t)a.H);
    T.b = (long long)bb;
    T.lay = (int)fdiv(bb, a.fd_bpl);
    T.bs = (int)(bb - (uint32_t)T.lay * (uint32_t)a.bpl);
    T.g = (int)fdiv((uint32_t)T.h, a.fd_hpg);
    T.row0 = ptile * kRows;
    T.rows = min(kRows, a.P - T.row0);
    long long sb = T.b;
    T.ok = true;
    if (POOL) {  // layer l's pool is states[l]: [nslots] sequence states
        int s = T.bs;
        if (a.slot != nullptr) {
            s = __ldg(a.slot + T.bs);
            T.ok = s >= 0 && s < a.nslots;
            if (!T.ok) s = 0;  // an invalid slot reads slot 0 (in bounds) and writes nothing
        }
        sb = (long long)T.lay * a.nslots + s;
    }
    T.sbase = (sb * a.H + T.h) * (long long)a.P * N;
    return T;
}

// Accepted prefix j of sequence b against a block of kref tokens: an
// out-of-range value counts as 0 and is reported.
__device__ __forceinline__ int accepted(const Args &a, long long b, int kref) {
    if (a.accept_len == nullptr) return kref;
    const int j = __ldg(a.accept_len + b);
    if (j < 0 || j > kref) {
        if (threadIdx.x == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_BAD_ACCEPT_LEN);
        return 0;
    }
    return j;
}

// Staged chunk of one phase: where its arrays live in shared memory.
struct StagedOffsets {
    int B, C, U, Dx, Abar, Cs, W, Xch;  // C, Dx, Cs, W, Xch: verify phase only
};

// dt values one thread needs to stage a chunk: the token of its x item
// (thread tid < kTC * ROWS / 8 handles rows 8 (tid % (ROWS / 8)) .. + 7 of token
// tid / (ROWS / 8)) and, for lane l of the last warp, token l (Abar,
// cumulative dt). Loaded one tile ahead so that their latency hides behind
// the previous tile's work.
struct ChunkDt {
    float x, tok;
};

template <typename Tin, int N>
__device__ __forceinline__ ChunkDt load_chunk_dt(const Args &a, const Block &blk, const Tile &T, int t0, int tc) {
    constexpr int XPT = Geo<N>::kRows / 8;
    const Tin *dtp = static_cast<const Tin *>(blk.dt);
    const int tid = threadIdx.x;
    const long long bt0 = T.b * blk.K + t0;
    ChunkDt d;
    const int tx = tid / XPT;
    d.x = (tid < kTC * XPT && tx < tc) ? ld1(dtp + (bt0 + tx) * a.H + T.h) : 0.f;
    const int lt = tid - (kThreads - 32);  // token lane of the last warp
    d.tok = (lt >= 0 && lt < tc) ? ld1(dtp + (bt0 + lt) * a.H + T.h) : 0.f;
    return d;
}

// The x and B items of one thread for a replay chunk, loaded from global memory
// before the tile's state arrives (N <= 128: at most one item of each per thread).
template <typename Tin>
struct PreItems {
    Raw8<Tin> x, b;
};
template <typename Tin, int N>
__device__ __forceinline__ PreItems<Tin> load_items(const Args &a, const Block &blk, const Tile &T, int tc) {
    constexpr int XPT = Geo<N>::kRows / 8, BPT = N / 8;
    static_assert(kTC * BPT <= kThreads, "one B item per thread");
    const int tid = threadIdx.x;
    const long long bt0 = T.b * blk.K;
    PreItems<Tin> p;
    const int t = tid / XPT, r8 = tid % XPT;
    if (tid < kTC * XPT && t < tc)
        ld8(static_cast<const Tin *>(blk.x) + ((bt0 + t) * a.H + T.h) * a.P + T.row0 + 8 * r8, blk.vec_x,
            T.rows - 8 * r8, p.x);
    const int tb = tid / BPT, n8 = tid % BPT;
    if (tid < kTC * BPT && tb < tc)
        ld8(static_cast<const Tin *>(blk.B) + ((bt0 + tb) * a.G + T.g) * N + 8 * n8, blk.vec_bc, 8, p.b);
    return p;
}

// Convert one chunk of tc tokens into the staged fp32 arrays, from the raw
// rows in shared memory (FROM_RAW: offsets rawX / rawB / rawC) or from global
// memory. x items are 8 rows of one token (u = dt x and D x), B/C items 8
// columns of one token. Tokens tc .. kTC-1 of u and B are zeroed (they meet
// zero weights in the contractions over the chunk and must not be NaN). The last
// warp also forms Abar, cs_t = sum_{r<=t} dt_r and w_t = exp(A cs_t) (verify phase).
// PRE: the x / B items come from load_items, issued earlier (global memory).
template <typename Tin, int N, bool WANT_Y, bool FROM_RAW, bool PRE = false>
__device__ __forceinline__ void stage_chunk(const Args &a, const Block &blk, const Tile &T, int t0, int tc, float Ah,
                                            float Dh, const StagedOffsets &so, int rawX, int rawB, int rawC,
                                            const ChunkDt &dt, const PreItems<Tin> *pre = nullptr) {
    constexpr int ROWS = Geo<N>::kRows;
    constexpr int XPT = ROWS / 8;  // x items per token
    constexpr int BPT = N / 8;     // B/C items per token
    static_assert(kTC * XPT <= kThreads, "one x item per thread");
    const Tin *xp = static_cast<const Tin *>(blk.x);
    const Tin *Bp = static_cast<const Tin *>(blk.B);
    const Tin *Cp = static_cast<const Tin *>(blk.C);
    const int tid = threadIdx.x;
    const long long bt0 = T.b * blk.K + t0;  // (b, t0) in [batch][K]

    // x item: u = dt x and D x for 8 rows of one token; zeros past tc.
    if (tid < kTC * XPT) {
        const int t = tid / XPT, r8 = tid % XPT;
        float xv[8];
        const float dtv = dt.x;
        if (t < tc) {
            Raw8<Tin> r;
            const long long row = (bt0 + t) * a.H + T.h;
            if constexpr (PRE) r = pre->x;
            else if (FROM_RAW) lds8(sm<const Tin>(rawX) + t * ROWS + 8 * r8, r);
            else ld8(xp + row * a.P + T.row0 + 8 * r8, blk.vec_x, T.rows - 8 * r8, r);
            widen(r, xv);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (8 * r8 + e >= T.rows) xv[e] = 0.f;  // past the tile: never stored
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) xv[e] = 0.f;
        }
        float *u = sm<float>(so.U) + t * Geo<N>::kUS + 8 * r8;
        st4(u, ssm_input_scale(dtv, xv[0]), ssm_input_scale(dtv, xv[1]), ssm_input_scale(dtv, xv[2]),
            ssm_input_scale(dtv, xv[3]));
        st4(u + 4, ssm_input_scale(dtv, xv[4]), ssm_input_scale(dtv, xv[5]), ssm_input_scale(dtv, xv[6]),
            ssm_input_scale(dtv, xv[7]));
        if (WANT_Y) {
            float *dx = sm<float>(so.Dx) + t * Geo<N>::kDS + 8 * r8;
            st4(dx, __fmul_rn(Dh, xv[0]), __fmul_rn(Dh, xv[1]), __fmul_rn(Dh, xv[2]), __fmul_rn(Dh, xv[3]));
            st4(dx + 4, __fmul_rn(Dh, xv[4]), __fmul_rn(Dh, xv[5]), __fmul_rn(Dh, xv[6]), __fmul_rn(Dh, xv[7]));
        }
    }
    // B / C items: 8 columns = two 4-column chunks, each to its thread's slots.
    // B of tokens tc .. kTC-1 is zeroed (the state update contracts over all
    // kTC tokens with zero weights there).
#pragma unroll 1
    for (int i = tid; i < kTC * BPT; i += kThreads) {
        const int t = i / BPT, n8 = i % BPT;
        const long long off = ((bt0 + t) * a.G + T.g) * N + 8 * n8;
        const int tb = t * Geo<N>::kWPB * 4 * Geo<N>::kPad;
        const int p0 = tb + perm_index<N>(8 * n8), p1 = tb + perm_index<N>(8 * n8 + 4);
        if (t >= tc) {
            st_slots<N>(sm<float>(so.B) + p0, 0.f, 0.f, 0.f, 0.f);
            st_slots<N>(sm<float>(so.B) + p1, 0.f, 0.f, 0.f, 0.f);
            continue;
        }
        Raw8<Tin> r;
        float v[8];
        if constexpr (PRE) r = pre->b;
        else if (FROM_RAW) lds8(sm<const Tin>(rawB) + t * N + 8 * n8, r);
        else ld8(Bp + off, blk.vec_bc, 8, r);
        widen(r, v);
        st_slots<N>(sm<float>(so.B) + p0, v[0], v[1], v[2], v[3]);
        st_slots<N>(sm<float>(so.B) + p1, v[4], v[5], v[6], v[7]);
        if (WANT_Y) {
            if (FROM_RAW) lds8(sm<const Tin>(rawC) + t * N + 8 * n8, r);
            else ld8(Cp + off, blk.vec_bc, 8, r);
            widen(r, v);
            st_slots<N>(sm<float>(so.C) + p0, v[0], v[1], v[2], v[3]);
            st_slots<N>(sm<float>(so.C) + p1, v[4], v[5], v[6], v[7]);
        }
    }
    // Per token (the last warp, whose lanes carry no tile-copy work): Abar and,
    // for y, the cumulative dt and the decay w from the chunk start.
    const int lt = tid - (kThreads - 32);
    if (lt >= 0) {
        const float dtv = dt.tok;  // 0 for lt >= tc
        if (lt < tc) sm<float>(so.Abar)[lt] = ssm_decay(dtv, Ah);
        if (WANT_Y) {
            float cs = dtv;  // inclusive prefix sum over the chunk's tokens
#pragma unroll
            for (int o = 1; o < kTC; o <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, cs, o);
                if (lt >= o) cs += v;
            }
            if (lt < kTC) {
                sm<float>(so.Cs)[lt] = cs;
                sm<float>(so.W)[lt] = lt < tc ? expf(__fmul_rn(Ah, cs)) : 0.f;
            }
        }
    }
}

// Thread-local view: warp `wp` of the CTA, lane (g = lane / 4, tq = lane % 4).
struct Lane {
    int band, half, g, tq, lane;
};

// Load the thread's 2 x NC slots of the state tile from shared memory
// (row-major [ROWS][N]); slots of rows past `rows` read as 0. Rows g and
// g + 1 of a quarter warp sit on the same banks (rows are multiples of 128
// bytes apart), so lanes with odd g fetch their column chunks in an order
// rotated by one: the two rows' accesses land 16 banks apart and every
// 128-bit load is conflict-free. The values are put back in slot order after.
template <int N>
__device__ __forceinline__ void load_state(float2 (&hs)[2][Geo<N>::kNC / 2], const Lane &L, int rows) {
    using G = Geo<N>;
    constexpr int M = G::kNC / 4;  // 4-column chunks per thread and row
    const float *sS = sm<const float>(0);
    const int rot = (M > 1) ? (L.g & 1) : 0;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = L.band * 16 + L.g + 8 * rr;
        const float *row = sS + r * N + L.half * G::kNCW;
        float4 v[M];
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const int mm = (m + rot) & (M - 1);
            v[m] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < rows) v[m] = *reinterpret_cast<const float4 *>(row + 4 * (L.tq + 4 * mm));
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const float4 w = rot ? v[(m + M - 1) & (M - 1)] : v[m];
            hs[rr][2 * m] = make_float2(w.x, w.y);
            hs[rr][2 * m + 1] = make_float2(w.z, w.w);
        }
    }
}

// Store the thread's slots of the state tile to global memory (rows past
// `rows` skipped). `sl` = state + sbase + row0 * N.
template <int N>
__device__ __forceinline__ void store_state(const float2 (&hs)[2][Geo<N>::kNC / 2], const Lane &L, float *sl,
                                            int rows) {
    using G = Geo<N>;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = L.band * 16 + L.g + 8 * rr;
        if (r < rows) {
            float *row = sl + (long long)r * N + L.half * G::kNCW;
#pragma unroll
            for (int m = 0; m < G::kNC / 4; ++m)
                __stcs(reinterpret_cast<float4 *>(row + 4 * (L.tq + 4 * m)),
                       make_float4(hs[rr][2 * m].x, hs[rr][2 * m].y, hs[rr][2 * m + 1].x, hs[rr][2 * m + 1].y));
        }
    }
}

// One recurrence step (staged token t): h <- Abar_t h + u_t[p] B_t^T.
template <int N>
__device__ __forceinline__ void recur_token(float2 (&hs)[2][Geo<N>::kNC / 2], const Lane &L, const StagedOffsets &so,
                                            int t) {
    using G = Geo<N>;
    constexpr int ROWS = G::kRows;
    const float abar = sm<const float>(so.Abar)[t];
    const float2 ab2 = make_float2(abar, abar);
    const float *urow = sm<const float>(so.U) + t * G::kUS + L.band * 16 + L.g;
    const float2 u0 = make_float2(urow[0], urow[0]);
    const float2 u1 = make_float2(urow[8], urow[8]);
    const float *bs = sm<const float>(so.B) + (t * G::kWPB * 4 + L.half * 4 + L.tq) * G::kPad;
#pragma unroll
    for (int m = 0; m < G::kNC / 4; ++m) {
        const float4 b = *reinterpret_cast<const float4 *>(bs + 4 * m);
        const float2 b01 = make_float2(b.x, b.y), b23 = make_float2(b.z, b.w);
        hs[0][2 * m] = ssm_update2(hs[0][2 * m], ab2, u0, b01);
        hs[0][2 * m + 1] = ssm_update2(hs[0][2 * m + 1], ab2, u0, b23);
        hs[1][2 * m] = ssm_update2(hs[1][2 * m], ab2, u1, b01);
        hs[1][2 * m + 1] = ssm_update2(hs[1][2 * m + 1], ab2, u1, b23);
    }
}

// The split of an fp32 operand for mma: x = hi + lo exactly in fp32, hi the
// tf32 truncation of x, |lo| < 2^-10 |x|; mma reads lo to tf32 precision, so
// the two products carry |error| < 2^-20 |x| per term. Exact inputs (bf16
// values) need only the high part.
struct Split {
    uint32_t hi, lo;
};
__device__ __forceinline__ Split split(float x) {
    Split s;
    s.hi = tf32_hi(x);
    s.lo = __float_as_uint(x - __uint_as_float(s.hi));
    return s;
}

// The state crossing staged tokens [0, tc) of a chunk, regrouped (the recurrence
// unrolled over the tokens):
//     h <- lambda h + sum_{s<tc} w_s u_s B_s^T,   lambda = prod_{s<tc} Abar_s,   w_s = prod_{s<r<tc} Abar_r.
// This thread's A-fragment tokens are tq and tq + 4 (w = 0 from tc on).
struct AdvW {
    float w0, w1, lam;
};
__device__ __forceinline__ AdvW adv_weights(const float *abar, int tq, int tc) {
    AdvW r{0.f, 0.f, 1.f};
#pragma unroll
    for (int t = kTC - 1; t >= 0; --t) {
        if (t < tc) {
            if (t == tq) r.w0 = r.lam;
            if (t == tq + 4) r.w1 = r.lam;
            r.lam = __fmul_rn(r.lam, abar[t]);
        }
    }
    return r;
}

// A fragment of w o u (rows g, g + 8 of the band; tokens tq, tq + 4), split
// into tf32 high and low parts.
struct AFrag {
    Split a0, a1, a2, a3;
};
template <int US>
__device__ __forceinline__ AFrag adv_frag(const float *U, const Lane &L, const AdvW &w) {
    const int r0 = L.band * 16 + L.g, r1 = r0 + 8, t0 = L.tq, t1 = L.tq + 4;
    return AFrag{split(__fmul_rn(w.w0, U[t0 * US + r0])), split(__fmul_rn(w.w0, U[t0 * US + r1])),
                 split(__fmul_rn(w.w1, U[t1 * US + r0])), split(__fmul_rn(w.w1, U[t1 * US + r1]))};
}

// The rank-tc term of one n-block, sum_s w_s u_s B_s^T, from zero (small
// parts first); bf16 B is exact in tf32, fp32 B is split as well.
template <typename Tin>
__device__ __forceinline__ void rank_term(float (&d)[4], const AFrag &a, float b0, float b1) {
    d[0] = d[1] = d[2] = d[3] = 0.f;
    if constexpr (sizeof(Tin) == 2) {
        mma_tf32(d, a.a0.lo, a.a1.lo, a.a2.lo, a.a3.lo, __float_as_uint(b0), __float_as_uint(b1));
        mma_tf32(d, a.a0.hi, a.a1.hi, a.a2.hi, a.a3.hi, __float_as_uint(b0), __float_as_uint(b1));
    } else {
        const Split c0 = split(b0), c1 = split(b1);
        mma_tf32(d, a.a0.lo, a.a1.lo, a.a2.lo, a.a3.lo, c0.hi, c1.hi);
        mma_tf32(d, a.a0.hi, a.a1.hi, a.a2.hi, a.a3.hi, c0.lo, c1.lo);
        mma_tf32(d, a.a0.hi, a.a1.hi, a.a2.hi, a.a3.hi, c0.hi, c1.hi);
    }
}

// Advance the register state over staged tokens [0, tc) on the tensor cores:
// one rank-8 mma.sync m16n8k8 tf32 product per n-block, then h <- lambda h +
// term (one fp32 fma, round to nearest). The thread's slot pair (2 nb,
// 2 nb + 1) of rows g and g + 8 is the D fragment of n-block nb under the
// column permutation of the staged B (logical column j of n-block nb is
// physical column 4 (j / 2) + 16 (nb / 2) + 2 (nb % 2) + j % 2, staged at row
// j / 2, slot 2 nb + j % 2), so no state moves. One warp per band (N <= 128).
template <typename Tin, int N>
__device__ __forceinline__ void advance_mma(float2 (&hs)[2][Geo<N>::kNC / 2], const Lane &L, const StagedOffsets &so,
                                            int tc) {
    using G = Geo<N>;
    static_assert(G::kWPB == 1, "one warp per band");
    const AdvW w = adv_weights(sm<const float>(so.Abar), L.tq, tc);
    const AFrag a = adv_frag<G::kUS>(sm<const float>(so.U), L, w);
    const float2 l2 = make_float2(w.lam, w.lam);
    const float *Bs = sm<const float>(so.B) + (L.g >> 1) * G::kPad + (L.g & 1);
    const float *b0p = Bs + L.tq * 4 * G::kPad, *b1p = Bs + (L.tq + 4) * 4 * G::kPad;
#pragma unroll
    for (int nb = 0; nb < G::kNC / 2; ++nb) {
        float d[4];
        rank_term<Tin>(d, a, b0p[2 * nb], b1p[2 * nb]);
        hs[0][nb] = __ffma2_rn(l2, hs[0][nb], make_float2(d[0], d[1]));
        hs[1][nb] = __ffma2_rn(l2, hs[1][nb], make_float2(d[2], d[3]));
    }
}

// The state after token jc - 1 of the staged chunk, written to global memory
// without changing the register state: each n-block's value is formed by
// exactly the arithmetic of advance_mma(jc), so the written state equals that
// of a block that ends at that token. `sl` = state + sbase + row0 * N.
template <typename Tin, int N>
__device__ __forceinline__ void commit_mma(const float2 (&hs)[2][Geo<N>::kNC / 2], const Lane &L,
                                           const StagedOffsets &so, int jc, float *sl, int rows) {
    using G = Geo<N>;
    static_assert(G::kWPB == 1, "one warp per band");
    const AdvW w = adv_weights(sm<const float>(so.Abar), L.tq, jc);
    const AFrag a = adv_frag<G::kUS>(sm<const float>(so.U), L, w);
    const float2 l2 = make_float2(w.lam, w.lam);
    const float *Bs = sm<const float>(so.B) + (L.g >> 1) * G::kPad + (L.g & 1);
    const float *b0p = Bs + L.tq * 4 * G::kPad, *b1p = Bs + (L.tq + 4) * 4 * G::kPad;
    const int r0 = L.band * 16 + L.g;
    float *row0 = sl + (long long)r0 * N + L.half * G::kNCW + 4 * L.tq, *row1 = row0 + 8LL * N;
#pragma unroll
    for (int nb = 0; nb < G::kNC / 2; ++nb) {
        float d[4];
        rank_term<Tin>(d, a, b0p[2 * nb], b1p[2 * nb]);
        // slot pair nb of rows g and g + 8: columns 4 (tq + 4 (nb / 2)) + 2 (nb % 2) + {0, 1}
        const int off = 16 * (nb >> 1) + 2 * (nb & 1);
        if (r0 < rows) __stcs(reinterpret_cast<float2 *>(row0 + off), __ffma2_rn(l2, hs[0][nb], make_float2(d[0], d[1])));
        if (r0 + 8 < rows)
            __stcs(reinterpret_cast<float2 *>(row1 + off), __ffma2_rn(l2, hs[1][nb], make_float2(d[2], d[3])));
    }
}

// y for the staged verify chunk (tc tokens, chunk start state hs):
//   y_t = w_t (C_t . h) + sum_{s<=t} L[t,s] (C_t . B_s) u_s + D x_t
// h . C^T and C . B^T on the tensor cores; y stored to ychunk + t * ystride + row.
template <typename Tin, int N>
__device__ __forceinline__ void chunk_y(const float2 (&hs)[2][Geo<N>::kNC / 2], const Lane &L,
                                        const StagedOffsets &so, int tc, float Ah, float *ychunk, long long ystride,
                                        int rows) {
    using G = Geo<N>;
    constexpr int ROWS = G::kRows;
    constexpr bool kExact = sizeof(Tin) == 2;  // bf16 B and C are exact tf32 values
    const float *Cs = sm<const float>(so.C) + (L.g * G::kWPB * 4 + L.half * 4 + L.tq) * G::kPad;
    const float *Bs = sm<const float>(so.B) + (L.g * G::kWPB * 4 + L.half * 4 + L.tq) * G::kPad;

    // Y0 = h . C^T (rows g, g+8; tokens 2tq, 2tq+1) and Gm = C . B^T (row g = token t,
    // columns 2tq, 2tq+1 = tokens s; rows g+8 of the mma are unused), over the warp's columns.
    // fp32 inputs: the two low-part products accumulate in yl, apart from the
    // high-part one, and are added in a fixed order after the loop.
    float yl[4] = {0.f, 0.f, 0.f, 0.f};
    float y0[4] = {0.f, 0.f, 0.f, 0.f};
    float gm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kb = 0; kb < G::kKB; ++kb) {
        const float2 c = *reinterpret_cast<const float2 *>(Cs + 2 * kb);
        const float2 bv = *reinterpret_cast<const float2 *>(Bs + 2 * kb);
        const Split h00 = split(hs[0][kb].x), h10 = split(hs[1][kb].x), h01 = split(hs[0][kb].y),
                    h11 = split(hs[1][kb].y);
        if constexpr (kExact) {
            const uint32_t c0 = __float_as_uint(c.x), c1 = __float_as_uint(c.y);
            mma_tf32(y0, h00.lo, h10.lo, h01.lo, h11.lo, c0, c1);
            mma_tf32(y0, h00.hi, h10.hi, h01.hi, h11.hi, c0, c1);
            mma_tf32(gm, c0, 0u, c1, 0u, __float_as_uint(bv.x), __float_as_uint(bv.y));
        } else {
            const Split c0 = split(c.x), c1 = split(c.y), b0 = split(bv.x), b1 = split(bv.y);
            mma_tf32(yl, h00.lo, h10.lo, h01.lo, h11.lo, c0.hi, c1.hi);
            mma_tf32(yl, h00.hi, h10.hi, h01.hi, h11.hi, c0.lo, c1.lo);
            mma_tf32(y0, h00.hi, h10.hi, h01.hi, h11.hi, c0.hi, c1.hi);
            mma_tf32(gm, c0.lo, 0u, c1.lo, 0u, b0.hi, b1.hi);
            mma_tf32(gm, c0.hi, 0u, c1.hi, 0u, b0.lo, b1.lo);
            mma_tf32(gm, c0.hi, 0u, c1.hi, 0u, b0.hi, b1.hi);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) y0[i] += yl[i];
    if constexpr (G::kWPB > 1) {
        // The band's second column half hands its partial Y0 and Gm to the first
        // through shared memory (a named barrier over the band's two warps).
        float *x = sm<float>(so.Xch) + (L.band * 32 + L.lane) * 8;
        if (L.half == 1) {
            st4(x, y0[0], y0[1], y0[2], y0[3]);
            x[4] = gm[0];
            x[5] = gm[1];
        }
        asm volatile("bar.sync %0, 64;" ::"r"(1 + L.band) : "memory");
        if (L.half == 1) return;
        y0[0] += x[0]; y0[1] += x[1]; y0[2] += x[2]; y0[3] += x[3];
        gm[0] += x[4];
        gm[1] += x[5];
    }
    // W[t][s] = L[t,s] Gm[t][s] for s <= t < tc (else 0); this lane holds t = g, s = 2tq, 2tq+1.
    const float *cs = sm<const float>(so.Cs);
    float w2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int t = L.g, s = 2 * L.tq + e;
        w2[e] = (s <= t && t < tc) ? expf(__fmul_rn(Ah, cs[t] - cs[s])) * gm[e] : 0.f;
    }
    // The intra-chunk term U . W^T: B fragment b0 = W[g][tq], b1 = W[g][tq + 4],
    // gathered from the quad holding row g.
    const int src0 = (L.lane & ~3) | (L.tq >> 1), src1 = src0 + 2;
    const float x0 = __shfl_sync(0xffffffffu, w2[0], src0), x1 = __shfl_sync(0xffffffffu, w2[1], src0);
    const float z0 = __shfl_sync(0xffffffffu, w2[0], src1), z1 = __shfl_sync(0xffffffffu, w2[1], src1);
    const Split wb0 = split((L.tq & 1) ? x1 : x0), wb1 = split((L.tq & 1) ? z1 : z0);
    const float *U = sm<const float>(so.U) + L.band * 16 + L.g;
    const Split ua0 = split(U[L.tq * G::kUS]), ua1 = split(U[L.tq * G::kUS + 8]),
                ua2 = split(U[(L.tq + 4) * G::kUS]), ua3 = split(U[(L.tq + 4) * G::kUS + 8]);
    // y = w (.) Y0 + U W^T
    const float *wt = sm<const float>(so.W);
    float d[4];
    d[0] = y0[0] * wt[2 * L.tq];
    d[1] = y0[1] * wt[2 * L.tq + 1];
    d[2] = y0[2] * wt[2 * L.tq];
    d[3] = y0[3] * wt[2 * L.tq + 1];
    mma_tf32(d, ua0.lo, ua1.lo, ua2.lo, ua3.lo, wb0.hi, wb1.hi);
    mma_tf32(d, ua0.hi, ua1.hi, ua2.hi, ua3.hi, wb0.lo, wb1.lo);
    mma_tf32(d, ua0.hi, ua1.hi, ua2.hi, ua3.hi, wb0.hi, wb1.hi);
    // + D x, store rows g, g + 8 for tokens 2tq, 2tq + 1.
    const float *Dx = sm<const float>(so.Dx);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = 2 * L.tq + (i & 1), r = L.band * 16 + L.g + 8 * (i >> 1);
        if (t < tc && r < rows) __stcs(ychunk + t * ystride + r, d[i] + Dx[t * G::kDS + r]);
    }
}

// Is there work for tile t? Only commit-only launches skip tiles (j = 0 or
// an invalid j: nothing to replay, nothing to write).
template <int F>
__device__ __forceinline__ long long next_work(const Args &a, long long t) {
    if constexpr (Flav<F>::kBase == kCommit) {
        if (a.accept_len == nullptr) return t;  // every token of every sequence
        const long long per_b = (long long)a.H * a.ptiles;
        for (; t < a.ntiles; t += gridDim.x) {
            const int j = __ldg(a.accept_len + (t / per_b) % a.bpl);  // every layer shares accept_len
            if (j > 0 && j <= a.rep.K) return t;
            if (j != 0 && threadIdx.x == 0 && a.dev_status != nullptr)
                atomicOr(a.dev_status, SSM_STATUS_BAD_ACCEPT_LEN);
        }
        return a.ntiles;
    } else {
        return t;
    }
}

#ifndef SSM_REGCAP
#define SSM_REGCAP 128
#endif
// Register budget per thread (resident CTAs of 128 threads = 65536 / (128 x cap)),
// or that of the CTAs the flavour's shared memory lets reside, if fewer.
template <typename Tin, int N, int F>
constexpr int min_blocks() {
    constexpr int by_regs = 65536 / SSM_REGCAP / kThreads > 0 ? 65536 / SSM_REGCAP / kThreads : 1;
    constexpr int by_smem = (228 * 1024) / (Lay<Tin, N, F>::kBytes + 1024);
    return by_smem < 1 ? 1 : (by_smem < by_regs ? by_smem : by_regs);
}

template <typename Tin, int N, int F>
__global__ void __launch_bounds__(kThreads, (min_blocks<Tin, N, F>())) ssm_tile_kernel(const Args a) {
    using G = Geo<N>;
    using FL = Flav<F>;
    using LY = Lay<Tin, N, F>;
    constexpr int ROWS = G::kRows;
    constexpr int E = (int)sizeof(Tin);
    __shared__ uint64_t bar;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    Lane L;
    L.band = warp / G::kWPB;
    L.half = warp % G::kWPB;
    L.g = lane >> 2;
    L.tq = lane & 3;
    L.lane = lane;
    const StagedOffsets sV{LY::kVB, LY::kVC, LY::kVU, LY::kVDx, LY::kVAbar, LY::kVCs, LY::kVW, LY::kXch};
    const StagedOffsets sR{LY::kRB, LY::kRB, LY::kRU, LY::kRU, LY::kRAbar, LY::kRAbar, LY::kRAbar, LY::kRAbar};

    // Launched with programmatic dependence (grids of no more CTAs than SMs), this grid may be resident
    // while the previous kernel of the stream finishes: nothing global is touched before that kernel has
    // completed and its writes are visible. Without that launch attribute both instructions do nothing.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    long long t = next_work<F>(a, blockIdx.x);
    if (t >= a.ntiles) return;  // uniform over the CTA

    // A tile streams into shared memory as one transaction on `bar`: the state
    // rows and, where the layout allows, the raw x / B / C rows of the first
    // chunk of the verify phase, or of the replay phase in the commit-only
    // flavour. The copies [state, replay x rows, replay B rows, verify x rows,
    // verify B rows, verify C rows] are spread over the warps
    // (copy k to lane k / 4 of warp k % 4); plan() works out this lane's copy
    // (while the state registers are free), issue() fires it, and lane 0 of
    // warp 0 announces the transaction's total bytes (a completion may arrive
    // before the announcement: the mbarrier's transaction count goes negative
    // meanwhile, and the phase cannot complete before the announcement).
    struct Plan {
        const void *src;
        uint32_t dst, bytes;  // dst: offset into the dynamic shared memory; bytes 0: none
        uint32_t total;
    };
    auto plan = [&](const Tile &T, long long tt, int buf) {
        Plan pl{nullptr, 0u, 0u, 0u};
        if (tt >= a.ntiles) return pl;
        const int tcR = LY::RR && a.rep.tma ? min(accepted(a, T.bs, a.rep.K), kTC) : 0;
        const int tcV = FL::kVerifyPhase && a.ver.tma ? min(a.ver.K, kTC) : 0;
        const uint32_t xrow = (uint32_t)T.rows * E, bcrow = (uint32_t)N * E;
        pl.total = (FL::kZero ? 0u : (uint32_t)T.rows * N * 4) + tcR * (xrow + bcrow) + tcV * (xrow + 2 * bcrow);
        const int ncopy = 1 + 2 * tcR + 3 * tcV;
        const int i = warp + 4 * lane;
        if (i >= ncopy) return pl;
        if (i == 0) {
            if (FL::kZero) return pl;  // no state copy
            pl.src = a.state_in + T.sbase + (long long)T.row0 * N;
            pl.dst = LY::kState;
            pl.bytes = (uint32_t)T.rows * N * 4;
            return pl;
        }
        int k = i - 1;
        const bool rep = k < 2 * tcR;
        if (!rep) k -= 2 * tcR;
        const int per = rep ? max(tcR, 1) : max(tcV, 1);
        const int kind = k / per;  // 0: x row, 1: B row, 2: C row
        const int tok = k % per;
        const long long bt = T.b * (rep ? a.rep.K : a.ver.K) + tok;
        if (kind == 0) {
            pl.src = static_cast<const Tin *>(rep ? a.rep.x : a.ver.x) + (bt * a.H + T.h) * a.P + T.row0;
            pl.dst = LY::kRaw + buf * LY::kRawBytes + (rep ? LY::oRx : LY::oVx) + tok * ROWS * E;
            pl.bytes = xrow;
        } else {
            const void *bc = rep ? a.rep.B : (kind == 1 ? a.ver.B : a.ver.C);
            pl.src = static_cast<const Tin *>(bc) + (bt * a.G + T.g) * N;
            pl.dst = LY::kRaw + buf * LY::kRawBytes + (rep ? LY::oRB : (kind == 1 ? LY::oVB : LY::oVC)) + tok * N * E;
            pl.bytes = bcrow;
        }
        return pl;
    };
    auto issue = [&](const Plan &pl) {
        if (tid == 0) mbar_arrive_expect_tx(&bar, pl.total);
        if (pl.bytes != 0) {
            if (pl.dst == LY::kState) bulk_load_once(ssm_smem + pl.dst, pl.src, pl.bytes, &bar);
            else bulk_load(ssm_smem + pl.dst, pl.src, pl.bytes, &bar);
        }
    };

    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    Tile Tcur = decode<FL::kPool>(a, t, ROWS, N);  // each tile is decoded once, a tile ahead
    issue(plan(Tcur, t, 0));

    // Per-tile scalars and the dt values of the first chunks, loaded one tile
    // ahead (their latency hides behind the previous tile's work).
    struct TileIn {
        float Ah, Dh;
        int jr, jw;  // tokens replayed; verify token after which the state is written (-1: none)
        ChunkDt dR, dV;
    };
    auto load_in = [&](const Tile &T, long long tt) {
        TileIn in{0.f, 0.f, 0, -1, {0.f, 0.f}, {0.f, 0.f}};
        if (tt >= a.ntiles) return in;
        in.Ah = __ldg(a.A + T.lay * a.H + T.h);
        if (FL::kVerifyPhase) in.Dh = __ldg(a.D + T.lay * a.H + T.h);
        if (FL::kReplay) in.jr = accepted(a, T.bs, a.rep.K);
        if (FL::kWriteInVerify) in.jw = accepted(a, T.bs, a.ver.K) - 1;
        if constexpr (FL::kReplay) in.dR = load_chunk_dt<Tin, N>(a, a.rep, T, 0, min(in.jr, kTC));
        if constexpr (FL::kVerifyPhase) in.dV = load_chunk_dt<Tin, N>(a, a.ver, T, 0, min(a.ver.K, kTC));
        return in;
    };
    TileIn cur = load_in(Tcur, t);

    uint32_t parity = 0;  // mbarrier phase; raw buffer of the current tile = parity
    while (t < a.ntiles) {
        const Tile T = Tcur;
        const float Ah = cur.Ah, Dh = cur.Dh;
        const int jr = cur.jr, jw = cur.jw;
        const int tcR0 = min(jr, kTC), tcV0 = FL::kVerifyPhase ? min(a.ver.K, kTC) : 0;
        const ChunkDt dR = cur.dR, dV = cur.dV;
        const long long tn = next_work<F>(a, t + gridDim.x);
        Tile Tn = T;
        if (tn < a.ntiles) Tn = decode<FL::kPool>(a, tn, ROWS, N);
        const Plan next = plan(Tn, tn, (int)(parity ^ 1u));
        cur = load_in(Tn, tn);
        Tcur = Tn;

        // Deferred-commit flavours at N <= 128: the replay chunk's x / B items are loaded
        // before the wait, while no state registers are live, so their latency overlaps it.
        constexpr bool kPre = FL::kReplay && FL::kVerifyPhase && kTC * (N / 8) <= kThreads;
        PreItems<Tin> pre;
        if constexpr (kPre)
            if (jr > 0) pre = load_items<Tin, N>(a, a.rep, T, tcR0);
        // Wait for the tile's bulk copies; the state tile goes to registers.
        const bool ok = mbar_wait_bounded(&bar, parity);
        float2 hs[2][G::kNC / 2];
        if constexpr (FL::kZero) {
#pragma unroll
            for (int rr = 0; rr < 2; ++rr)
#pragma unroll
                for (int m = 0; m < G::kNC / 2; ++m) hs[rr][m] = make_float2(0.f, 0.f);
        } else {
            load_state<N>(hs, L, T.rows);
        }
        // Every thread is done with the state tile and with the previous tile's
        // staged inputs; the vote makes a timeout a CTA-wide decision.
        if (__syncthreads_or(!ok)) {
            if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_TIMEOUT);
            mbar_wait_bounded(&bar, parity);  // drain the copies still in flight, bounded
            return;
        }
        if (tn < a.ntiles) {
            fence_proxy_async_smem();
            issue(next);
        }
        // Stage the first chunk of each phase: from this tile's raw buffer, or
        // from global memory where the layout does not allow bulk copies (and,
        // in the deferred-commit flavours, the replay chunk from the items loaded
        // before the wait; their verify chunk is staged after the replay).
        const int raw = LY::kRaw + (int)parity * LY::kRawBytes;
        if constexpr (FL::kReplay) {
            if (jr > 0) {
                if (LY::RR && a.rep.tma)
                    stage_chunk<Tin, N, false, true>(a, a.rep, T, 0, tcR0, Ah, 0.f, sR, raw + LY::oRx, raw + LY::oRB,
                                                     raw + LY::oRB, dR);
                else if constexpr (kPre)
                    stage_chunk<Tin, N, false, false, true>(a, a.rep, T, 0, tcR0, Ah, 0.f, sR, 0, 0, 0, dR, &pre);
                else
                    stage_chunk<Tin, N, false, false>(a, a.rep, T, 0, tcR0, Ah, 0.f, sR, 0, 0, 0, dR);
            }
        }
        if constexpr (FL::kVerifyPhase && !FL::kReplay) {
            if (a.ver.tma)
                stage_chunk<Tin, N, true, true>(a, a.ver, T, 0, tcV0, Ah, Dh, sV, raw + LY::oVx, raw + LY::oVB,
                                                raw + LY::oVC, dV);
            else
                stage_chunk<Tin, N, true, false>(a, a.ver, T, 0, tcV0, Ah, Dh, sV, 0, 0, 0, dV);
        }
        parity ^= 1u;
        __syncthreads();  // staged inputs visible
        if constexpr (FL::kPool) {
            if (!T.ok) {  // no valid pool slot: neither y nor the state is written
                if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_BAD_SLOT);
                t = tn;
                continue;
            }
        }

        float *sl = (a.state != nullptr) ? a.state + T.sbase + (long long)T.row0 * N : nullptr;

        if constexpr (FL::kReplay) {
            // Replay phase: advance over tokens 0 .. jr-1 of the replay block, then commit h_jr.
            for (int t0 = 0; t0 < jr; t0 += kTC) {
                const int tc = min(kTC, jr - t0);
                if (t0 > 0) {
                    const ChunkDt d = load_chunk_dt<Tin, N>(a, a.rep, T, t0, tc);
                    __syncthreads();
                    stage_chunk<Tin, N, false, false>(a, a.rep, T, t0, tc, Ah, 0.f, sR, 0, 0, 0, d);
                    __syncthreads();
                }
                if constexpr (G::kWPB == 1) {
                    advance_mma<Tin, N>(hs, L, sR, tc);
                } else {
#pragma unroll 1
                    for (int s = 0; s < tc; ++s) recur_token<N>(hs, L, sR, s);
                }
            }
            if (jr > 0) store_state<N>(hs, L, sl, T.rows);
        }
        if constexpr (FL::kReplay && FL::kVerifyPhase) {
            // the verify phase's first chunk, into the arrays the replay has finished reading
            __syncthreads();
            if (a.ver.tma)
                stage_chunk<Tin, N, true, true>(a, a.ver, T, 0, tcV0, Ah, Dh, sV, raw + LY::oVx, raw + LY::oVB,
                                                raw + LY::oVC, dV);
            else
                stage_chunk<Tin, N, true, false>(a, a.ver, T, 0, tcV0, Ah, Dh, sV, 0, 0, 0, dV);
            __syncthreads();
        }

        if constexpr (FL::kVerifyPhase) {
            const int K = a.ver.K;
            float *ytile = a.y + (T.b * K * a.H + T.h) * (long long)a.P + T.row0;
            const long long ystride = (long long)a.H * a.P;
            for (int t0 = 0; t0 < K; t0 += kTC) {
                const int tc = min(kTC, K - t0);
                if (t0 > 0) {
                    const ChunkDt d = load_chunk_dt<Tin, N>(a, a.ver, T, t0, tc);
                    __syncthreads();
                    stage_chunk<Tin, N, true, false>(a, a.ver, T, t0, tc, Ah, Dh, sV, 0, 0, 0, d);
                    __syncthreads();
                }
                chunk_y<Tin, N>(hs, L, sV, tc, Ah, ytile + t0 * ystride, ystride, T.rows);
                // Advance the state by the recurrence as far as it is needed: through the
                // chunk when more chunks follow, else up to the committed token.
                const bool more = t0 + tc < K;
                if constexpr (G::kWPB == 1) {
                    // jc: the committed state is the one after token jc - 1 of this chunk
                    const int jc = (FL::kWriteInVerify && jw >= t0 && jw < t0 + tc) ? jw - t0 + 1 : 0;
                    if (more && jc > 0 && jc < tc) {
                        commit_mma<Tin, N>(hs, L, sV, jc, sl, T.rows);
                        advance_mma<Tin, N>(hs, L, sV, tc);
                    } else {
                        const int adv = more ? tc : jc;
                        if (adv > 0) advance_mma<Tin, N>(hs, L, sV, adv);
                        if (jc > 0) store_state<N>(hs, L, sl, T.rows);
                    }
                } else {
                    int steps = 0;
                    if (more) steps = tc;
                    else if (FL::kWriteInVerify && jw >= t0) steps = jw - t0 + 1;
#pragma unroll 1
                    for (int s = 0; s < steps; ++s) {
                        recur_token<N>(hs, L, sV, s);
                        if (FL::kWriteInVerify && t0 + s == jw) store_state<N>(hs, L, sl, T.rows);
                    }
                }
            }
        }
        t = tn;
    }
}

// Failure-detection self-test: one warp waits, with the bounded wait of the
// tile kernel, on an mbarrier phase whose announced bytes never arrive (no copy
// is issued), and reports the timeout. Nothing but *status is touched.
__global__ void ssm_wait_timeout_kernel(uint32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(&bar, 16u);
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded(&bar, 0u);
    if (__any_sync(0xffffffffu, !ok) && threadIdx.x == 0 && status != nullptr) atomicOr(status, SSM_STATUS_TIMEOUT);
}


// ----------------------------------------------------------------------------- prefill kernels

// Chunked prefill, first pass on the tensor cores: the state a chunk of L
// tokens leaves when it starts from h = 0 -- the recurrence unrolled over
// the chunk,
//     S[p][n] = sum_s w_s u_s[p] B_s[n],   w_s = prod_{r > s} Abar_r,   u_s = dt_s x_s,
// -- as one contraction over the chunk's tokens, (w o U) (rows x L) times
// B (L x N), on mma.sync m16n8k8 tf32 with fp32 accumulation. w o U is split
// into tf32 high and low parts so that the products keep fp32 accuracy; bf16
// B is exact in tf32, fp32 B is split as well. One 64-row tile of one head
// of one chunk per CTA (16 rows per warp; a thread's accumulators are the
// state-register layout of the tile kernel).
constexpr int kCSRows = 64;
constexpr int kCSMaxL = 128;

struct CSArgs {
    const void *x, *B, *dt;  // chunk v = tokens v*L .. v*L + L - 1 of the [batch][T] layouts
    const float *A;
    float *ws;               // [chunks][H][P][N]
    float *lam;              // [chunks][H]: lambda = the product of the chunk's Abar, for the scan
    uint32_t *dev_status;    // nullable (the tensor-memory kernel's bounded wait)
    int H, P, G, L, ptiles;  // ptiles: tiles of a chunk (P / 64 per head; H P / 128 on the tensor cores)
};

template <typename Tin, int N>
struct CSLay {
    static constexpr int kXPad = kCSRows + 8;  // x staged token-major, rows padded: conflict-free fragments
    static constexpr int kBPad = N + 8;
    static constexpr int kX = 0;
    static constexpr int kB = kX + kCSMaxL * kXPad * (int)sizeof(Tin);
    static constexpr int kW = kB + kCSMaxL * kBPad * (int)sizeof(Tin);
    static constexpr int kW2 = kW + kCSMaxL * 4;  // second buffer of the suffix-product scan
    static constexpr int kDt = kW2 + kCSMaxL * 4;
    static constexpr int kBytes = kDt + kCSMaxL * 4;
    static_assert(kB % 16 == 0 && (kXPad * sizeof(Tin)) % 16 == 0 && (kBPad * sizeof(Tin)) % 16 == 0, "alignment");
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ float sval(const float *p) { return *p; }
__device__ __forceinline__ float sval(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

template <typename Tin, int N>
__global__ void __launch_bounds__(128) ssm_chunk_state_kernel(const CSArgs a) {
    using LY = CSLay<Tin, N>;
    constexpr int NB = N / 8;
    constexpr int VW = 16 / (int)sizeof(Tin);  // elements per 16-byte vector
    Tin *sx = sm<Tin>(LY::kX);
    Tin *sb = sm<Tin>(LY::kB);
    float *sw = sm<float>(LY::kW), *sw2 = sm<float>(LY::kW2), *sdt = sm<float>(LY::kDt);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, tq = lane & 3;
    const long long t = blockIdx.x;
    const int ptile = (int)(t % a.ptiles);
    const long long vh = t / a.ptiles;
    const int h = (int)(vh % a.H);
    const long long v = vh / a.H;
    const int gi = h / (a.H / a.G);
    const int row0 = ptile * kCSRows;
    const int L = a.L;
    const float Ah = __ldg(a.A + h);
    const Tin *x = static_cast<const Tin *>(a.x);
    const Tin *Bp = static_cast<const Tin *>(a.B);
    const Tin *dtp = static_cast<const Tin *>(a.dt);

    // stage the chunk's x rows (this tile's 64 rows) and B rows, 16 bytes at a time
    for (int i = tid; i < L * (kCSRows / VW); i += 128) {
        const int s = i / (kCSRows / VW), q = i % (kCSRows / VW);
        cp_async16(sx + s * LY::kXPad + q * VW, x + ((v * L + s) * a.H + h) * (long long)a.P + row0 + q * VW);
    }
    for (int i = tid; i < L * (N / VW); i += 128) {
        const int s = i / (N / VW), q = i % (N / VW);
        cp_async16(sb + s * LY::kBPad + q * VW, Bp + ((v * L + s) * a.G + gi) * (long long)N + q * VW);
    }
    // dt and the suffix products w_s = prod_{r > s} Abar_r (a fixed product tree)
    float abar0 = 1.f;
    if (tid < L) {
        const float d = ld1(dtp + (v * L + tid) * a.H + h);
        sdt[tid] = d;
        sw[tid] = tid + 1 < L ? ssm_decay(ld1(dtp + (v * L + tid + 1) * a.H + h), Ah) : 1.f;
        if (tid == 0) abar0 = ssm_decay(d, Ah);
    }
    __syncthreads();
    float *cur = sw, *nxt = sw2;
    for (int d = 1; d < L; d <<= 1) {
        if (tid < L) nxt[tid] = tid + d < L ? __fmul_rn(cur[tid], cur[tid + d]) : cur[tid];
        __syncthreads();
        float *tmp = cur;
        cur = nxt;
        nxt = tmp;
    }
    // the chunk's lambda = Abar_0 w_0, once per chunk and head (the head's first row tile)
    if (tid == 0 && ptile == 0) a.lam[v * a.H + h] = __fmul_rn(abar0, cur[0]);
    cp_async_wait_all();
    __syncthreads();

    float acc[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.f;
    const int r0 = warp * 16 + g, r1 = r0 + 8;
    for (int kb = 0; kb < L / 8; ++kb) {
        const int s0 = kb * 8 + tq, s1 = s0 + 4;
        const float w0 = cur[s0], w1 = cur[s1], d0 = sdt[s0], d1 = sdt[s1];
        const Split a0 = split(__fmul_rn(w0, ssm_input_scale(d0, sval(sx + s0 * LY::kXPad + r0))));
        const Split a1 = split(__fmul_rn(w0, ssm_input_scale(d0, sval(sx + s0 * LY::kXPad + r1))));
        const Split a2 = split(__fmul_rn(w1, ssm_input_scale(d1, sval(sx + s1 * LY::kXPad + r0))));
        const Split a3 = split(__fmul_rn(w1, ssm_input_scale(d1, sval(sx + s1 * LY::kXPad + r1))));
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
            const float b0 = sval(sb + s0 * LY::kBPad + nb * 8 + g), b1 = sval(sb + s1 * LY::kBPad + nb * 8 + g);
            if constexpr (sizeof(Tin) == 2) {  // bf16 values are exact in tf32
                const uint32_t e0 = __float_as_uint(b0), e1 = __float_as_uint(b1);
                mma_tf32(acc[nb], a0.hi, a1.hi, a2.hi, a3.hi, e0, e1);
                mma_tf32(acc[nb], a0.lo, a1.lo, a2.lo, a3.lo, e0, e1);
            } else {
                const Split c0 = split(b0), c1 = split(b1);
                mma_tf32(acc[nb], a0.hi, a1.hi, a2.hi, a3.hi, c0.hi, c1.hi);
                mma_tf32(acc[nb], a0.lo, a1.lo, a2.lo, a3.lo, c0.hi, c1.hi);
                mma_tf32(acc[nb], a0.hi, a1.hi, a2.hi, a3.hi, c0.lo, c1.lo);
            }
        }
    }
    float *out = a.ws + ((v * a.H + h) * (long long)a.P + row0) * N;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int c = nb * 8 + 2 * tq;
        *reinterpret_cast<float2 *>(out + (long long)r0 * N + c) = make_float2(acc[nb][0], acc[nb][1]);
        *reinterpret_cast<float2 *>(out + (long long)r1 * N + c) = make_float2(acc[nb][2], acc[nb][3]);
    }
}

// The same first pass on the 5th-generation tensor cores (tcgen05), for bf16
// inputs, N = 128, L = 128 and 128-row tiles: one CTA computes
// S[p][n] = sum_s (w_s u_s[p]) B_s[n] for 128 rows of one chunk as an
// M = 128, N = 128, K = 128 product accumulated in tensor memory. The rows
// are 128 consecutive rows h P + p of the chunk's H P: of one head, or at
// P = 64 of two heads of one group (B is shared, w and dt are per head).
//  * Operands in shared memory, K-major (token index contiguous), no swizzle:
//    8-row x 16-byte core matrices; element (row r, token s) of an operand
//    sits at byte (r / 8) * 2048 + (s / 8) * 128 + (r % 8) * 16 + (s % 8) * 2;
//    the descriptor's leading offset is the token stride (128), its stride
//    offset the row stride (2048). x and B arrive row-contiguous per token,
//    so each thread transposes one 8 x 8 block of each in registers.
//  * w o U is formed in fp32 by the arithmetic of ssm_chunk_state_kernel and
//    split into two bf16 parts a1 + a2 (a1 = bf16(a), a2 = bf16(a - a1):
//    16 significant bits, |a - a1 - a2| <= 2^-18 |a|); B is bf16 and exact.
//    2 parts x 8 MMAs of K = 16 tokens (tcgen05.mma kind::f16, bf16 x bf16,
//    fp32 accumulation), issued by one thread; tcgen05.commit signals an
//    mbarrier, waited on with a time limit. 99 KB of shared memory: two
//    CTAs of 256 threads per SM.
//  * Row p of the accumulator is tensor-memory lane p: warps w and w + 4
//    read rows 32 (w % 4) .. + 31 (each half of the columns) with tcgen05.ld.
constexpr int kTCRows = 128;
constexpr int kTCParts = 2;
constexpr int kTCThreads = 256;
constexpr int kStagePitch = 132;  // floats per row of a 128 x 128 fp32 tile staged in shared memory (padded)
struct TCLay {
    static constexpr int kPart = 128 * 128 * 2;       // one bf16 operand: 128 rows x 128 tokens
    static constexpr int kA = 0;                      // w o U parts a1, a2
    static constexpr int kB = kA + kTCParts * kPart;  // B
    static constexpr int kW = kB + kPart;             // float[2][128]: per head of the tile (two at P = 64)
    static constexpr int kW2 = kW + 2 * 128 * 4;
    static constexpr int kDt = kW2 + 2 * 128 * 4;
    static constexpr int kBytes = kDt + 2 * 128 * 4;
};

// K-major operand: row r (M or N index), token (K index) k.
__device__ __forceinline__ uint32_t tck_off(int r, int k) {
    return (uint32_t)((r >> 3) * 2048 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}
__device__ __forceinline__ uint64_t tck_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) | ((uint64_t)(2048u >> 4) << 32) |
           ((uint64_t)1 << 46);
}
// kind::f16, fp32 accumulator, bf16 A and B, both K-major, M = N = 128.
constexpr uint32_t kTCIdescKK = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void tc_mma_i(uint32_t taddr, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(taddr),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, float (&f)[16]) {
    uint32_t u[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) f[i] = __uint_as_float(u[i]);
}
__device__ __forceinline__ uint32_t bf16_bits(__nv_bfloat16 v) { return (uint32_t)__bfloat16_as_ushort(v); }
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return bf16_bits(__float2bfloat16_rn(lo)) | (bf16_bits(__float2bfloat16_rn(hi)) << 16);
}
// 16-bit element e (0..7) of an 8-element row held as a uint4
__device__ __forceinline__ uint32_t u16_at(const uint4 &r, int e) {
    const uint32_t w = e < 4 ? (e < 2 ? r.x : r.y) : (e < 6 ? r.z : r.w);
    return (e & 1) ? (w >> 16) : (w & 0xFFFFu);
}

__global__ void __launch_bounds__(kTCThreads, 2) ssm_chunk_state_tc_kernel(const CSArgs a) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    unsigned char *sbytes = reinterpret_cast<unsigned char *>(ssm_smem);
    float *sw = sm<float>(TCLay::kW), *sw2 = sm<float>(TCLay::kW2), *sdt = sm<float>(TCLay::kDt);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // tile = 128 consecutive rows R = h P + p of the chunk's H P rows: one head, or two at P = 64 (same group)
    const long long t = blockIdx.x;
    const long long v = t / a.ptiles;
    const int R0 = (int)(t % a.ptiles) * kTCRows;
    const int h0 = R0 / a.P;
    const int nh = a.P >= kTCRows ? 1 : 2;
    const int gi = h0 / (a.H / a.G);
    constexpr int L = 128;
    const __nv_bfloat16 *x = static_cast<const __nv_bfloat16 *>(a.x);
    const __nv_bfloat16 *Bp = static_cast<const __nv_bfloat16 *>(a.B);
    const __nv_bfloat16 *dtp = static_cast<const __nv_bfloat16 *>(a.dt);

    // this thread's 8 x 8 blocks: tokens s0 .. s0+7 of rows p0 .. p0+7 (x) and of columns p0 .. p0+7 (B)
    const int bp = tid & 15, bs = tid >> 4, p0 = bp * 8, s0 = bs * 8;
    uint4 xr[8], br[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const long long bt = v * L + s0 + i;
        xr[i] = __ldg(reinterpret_cast<const uint4 *>(x + bt * a.H * (long long)a.P + R0 + p0));
        br[i] = __ldg(reinterpret_cast<const uint4 *>(Bp + (bt * a.G + gi) * 128LL + p0));
    }
    // dt and the suffix products w_s = prod_{r > s} Abar_r (the product tree of ssm_chunk_state_kernel), per head
    float abar0 = 1.f;
    if (tid < nh * L) {
        const int hh = h0 + (tid >> 7), s = tid & (L - 1);
        const float Ah = __ldg(a.A + hh);
        const float d = ld1(dtp + (v * L + s) * a.H + hh);
        sdt[tid] = d;
        sw[tid] = s + 1 < L ? ssm_decay(ld1(dtp + (v * L + s + 1) * a.H + hh), Ah) : 1.f;
        if (s == 0) abar0 = ssm_decay(d, Ah);
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {  // 128 columns of tensor memory: the fp32 accumulator, one lane per row
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 128;" ::"r"(smem_addr(&tmem_base))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // B transposed into its operand (row n = p0 + j, tokens s0 .. s0+7); row order rotated per lane
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int j = (k + lane) & 7;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) w[e / 2] = u16_at(br[e], j) | (u16_at(br[e + 1], j) << 16);
        *reinterpret_cast<uint4 *>(sbytes + TCLay::kB + tck_off(p0 + j, s0)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __syncthreads();
    float *cur = sw, *nxt = sw2;
    for (int d = 1; d < L; d <<= 1) {
        if (tid < nh * L) nxt[tid] = (tid & (L - 1)) + d < L ? __fmul_rn(cur[tid], cur[tid + d]) : cur[tid];
        __syncthreads();
        float *tmp = cur;
        cur = nxt;
        nxt = tmp;
    }
    // the chunk's lambda = Abar_0 w_0 of each head whose first row is in this tile (once per chunk and head)
    if (tid < nh * L && (tid & (L - 1)) == 0 && (long long)(h0 + (tid >> 7)) * a.P >= R0)
        a.lam[v * a.H + h0 + (tid >> 7)] = __fmul_rn(abar0, cur[tid]);
    // w o U in fp32, split into two bf16 parts, transposed into the A operands (row p0 + j, of head h0 + hf)
    const int hf = nh == 1 ? 0 : p0 / a.P;
    float wsv[8], dsv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        wsv[i] = cur[hf * L + s0 + i];
        dsv[i] = sdt[hf * L + s0 + i];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int j = (k + lane) & 7;
        uint32_t p1[4], p2[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            uint32_t w1[2], w2[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float xv = __uint_as_float(u16_at(xr[e + q], j) << 16);  // bf16 -> fp32, exact
                const float av = __fmul_rn(wsv[e + q], ssm_input_scale(dsv[e + q], xv));
                const __nv_bfloat16 b1 = __float2bfloat16_rn(av);
                w1[q] = bf16_bits(b1);
                w2[q] = bf16_bits(__float2bfloat16_rn(av - __bfloat162float(b1)));
            }
            p1[e / 2] = w1[0] | (w1[1] << 16);
            p2[e / 2] = w2[0] | (w2[1] << 16);
        }
        const uint32_t off = tck_off(p0 + j, s0);
        *reinterpret_cast<uint4 *>(sbytes + TCLay::kA + off) = make_uint4(p1[0], p1[1], p1[2], p1[3]);
        *reinterpret_cast<uint4 *>(sbytes + TCLay::kA + TCLay::kPart + off) = make_uint4(p2[0], p2[1], p2[2], p2[3]);
    }
    fence_proxy_async_smem();  // the operands written by the threads, visible to the tensor cores
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = tmem_base;
    if (tid == 0) {
        const uint32_t abase = smem_addr(sbytes + TCLay::kA), bbase = smem_addr(sbytes + TCLay::kB);
        for (int part = 0; part < kTCParts; ++part)
            for (int kk = 0; kk < L / 16; ++kk)
                tc_mma_i(taddr, tck_desc(abase + part * TCLay::kPart + kk * 256), tck_desc(bbase + kk * 256),
                         kTCIdescKK, (part | kk) != 0 ? 1u : 0u);
        tc_commit(&bar);
    }
    const bool ok = mbar_wait_bounded(&bar, 0u);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (__syncthreads_or(!ok)) {  // never on a healthy device: report, wait once more for the products
        if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_TIMEOUT);
        mbar_wait_bounded(&bar, 0u);
    } else {
        // the accumulator through shared memory (over the operands, which the products no longer read), so
        // that each warp then writes whole 512-byte rows
        const int r = (warp & 3) * 32 + lane, ch = (warp >> 2) * 64;
        float *stage = sm<float>(0);  // [128][kStagePitch]
        const uint32_t trow = taddr + ((uint32_t)((warp & 3) * 32) << 16);
#pragma unroll 1
        for (int c0 = ch; c0 < ch + 64; c0 += 16) {
            float f[16];
            tc_ld16(trow + c0, f);
#pragma unroll
            for (int k = 0; k < 16; k += 4)
                *reinterpret_cast<float4 *>(stage + r * kStagePitch + c0 + k) = make_float4(f[k], f[k + 1], f[k + 2], f[k + 3]);
        }
        __syncthreads();
        float *out = a.ws + (v * a.H * (long long)a.P + R0) * 128;
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {
            const int idx = it * kTCThreads + tid, row = idx >> 5, c4 = (idx & 31) * 4;
            *reinterpret_cast<float4 *>(out + (long long)row * 128 + c4) =
                *reinterpret_cast<const float4 *>(stage + row * kStagePitch + c4);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 128;" ::"r"(taddr) : "memory");
}

// Chunked prefill, output pass on the tensor cores (tcgen05), for the shapes
// of ssm_chunk_state_tc_kernel: y of every token of a 128-token chunk from the
// state H0 the chunk starts from, in the chunked (attention-like) form of the
// recurrence,
//     y_t = w_t (C_t . H0) + sum_{s<=t} exp(A (cs_t - cs_s)) dt_s (C_t . B_s) x_s + D x_t,
//     cs_t = sum_{r<=t} dt_r,   w_t = exp(A cs_t),
// for 128 rows p of one head (or 64: the tile's rows PR, where P is a multiple
// of 64 but not of 128, with Yi and Yc then N = 64 products). Three products
// accumulate in tensor memory:
//   Yi = C H0^T   (128 tokens x 128 rows, over 128 state channels; H0 split
//                  into two bf16 parts, C exact),
//   G  = C B^T    (128 x 128 tokens; bf16, exact inputs),
//   Yc = M X      (M[t][s] = G[t][s] exp(A (cs_t - cs_s)) dt_s for s <= t,
//                  else 0, split into two bf16 parts; x exact),
// and y = w_t Yi + Yc + D x. One CTA of 256 threads per (chunk, head,
// row tile), two CTAs per SM: three 32 KB operand buffers are reused
// phase by phase (C and B, then the low part of H0 over B, then M over H0
// and C with x over B), and Yc accumulates in G's tensor-memory columns once
// G has been read, so a CTA needs 97 KB of shared memory and 256 columns.
// Row t of every accumulator is tensor-memory lane t, read by warps w and
// w + 4 (each half of the columns). Every operand is K-major (leading offset
// 128, the K-direction stride; stride offset 2048): on this hardware a
// no-swizzle MN-major operand ran about ten times slower per instruction.
// x arrives row-contiguous per token, so each thread transposes one 8 x 8
// block in registers; the D x term reads x again from L2.
struct OutArgs {
    const void *x, *B, *C, *dt;  // [batch][T] layouts; chunk v = tokens v*128 .. v*128 + 127
    const float *A, *D;
    const float *ws;             // [chunks][H][P][N]: the state each chunk starts from
    const int32_t *vslot;        // nullable: chunk v writes no y where vslot[v] < 0
    float *y;                    // [batch][T][H][P]
    uint32_t *dev_status;
    int H, P, G, ptiles;
};

constexpr int kOutThreads = 256;
struct OutLay {
    static constexpr int kOp = 128 * 128 * 2;  // one bf16 operand, 128 x 128, K-major
    static constexpr int kP0 = 0;              // C, later M part 2
    static constexpr int kP1 = kP0 + kOp;      // B, then H0 part 2, then x (row p, token s)
    static constexpr int kP2 = kP1 + kOp;      // H0 part 1, later M part 1
    static constexpr int kCs = kP2 + kOp;      // float[128] cs_t
    static constexpr int kDt = kCs + 512;      // float[128] dt_t
    static constexpr int kBytes = kDt + 512;
};

template <int PR>  // rows of the tile: 128, or 64 (the products over rows are then N = 64)
__global__ void __launch_bounds__(kOutThreads, 2) ssm_chunk_out_tc_kernel(const OutArgs a) {
    static_assert(PR == 128 || PR == 64, "tile rows");
    constexpr uint32_t kIdescRows = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(PR >> 3) << 17) | ((128u >> 4) << 24);
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ float wsum[4];
    unsigned char *sb = reinterpret_cast<unsigned char *>(ssm_smem);
    float *scs = sm<float>(OutLay::kCs), *sdt = sm<float>(OutLay::kDt);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long tile = blockIdx.x;
    const int ptile = (int)(tile % a.ptiles);
    const long long vh = tile / a.ptiles;
    const int h = (int)(vh % a.H);
    const long long v = vh / a.H;
    const int gi = h / (a.H / a.G);
    const int row0 = ptile * PR;
    const float Ah = __ldg(a.A + h), Dh = __ldg(a.D + h);
    const bool write_y = a.vslot == nullptr || __ldg(a.vslot + v) >= 0;
    const __nv_bfloat16 *xg = static_cast<const __nv_bfloat16 *>(a.x);
    const __nv_bfloat16 *Bg = static_cast<const __nv_bfloat16 *>(a.B);
    const __nv_bfloat16 *Cg = static_cast<const __nv_bfloat16 *>(a.C);
    const __nv_bfloat16 *dtg = static_cast<const __nv_bfloat16 *>(a.dt);
    // warp task (8 consecutive rows x 4 consecutive 16-byte chunks), 8 per warp: conflict-free stores
    auto task_r = [&](int it) { return ((warp + 8 * it) & 15) * 8 + (lane & 7); };
    auto task_q = [&](int it) { return ((warp + 8 * it) >> 4) * 4 + (lane >> 3); };
    // the same over the tile's PR rows (PR / 16 tasks per warp)
    constexpr int kRG = PR / 8;
    auto htask_r = [&](int it) { return ((warp + 8 * it) % kRG) * 8 + (lane & 7); };
    auto htask_q = [&](int it) { return ((warp + 8 * it) / kRG) * 4 + (lane >> 3); };

    // C and B (K-major, row = token): straight into their operand layouts
#pragma unroll 4
    for (int it = 0; it < 8; ++it) {
        const int t = task_r(it), q = task_q(it);
        const long long bt = v * 128 + t;
        cp_async16(sb + OutLay::kP0 + tck_off(t, q * 8), Cg + (bt * a.G + gi) * 128LL + q * 8);
        cp_async16(sb + OutLay::kP1 + tck_off(t, q * 8), Bg + (bt * a.G + gi) * 128LL + q * 8);
    }
    // H0 (row p, K-major): high part into its operand now, low part kept packed for the second product
    const float *H0 = a.ws + ((v * a.H + h) * (long long)a.P + row0) * 128;
    uint4 hlo[PR / 16];
#pragma unroll
    for (int it = 0; it < PR / 16; ++it) {
        const float *src = H0 + htask_r(it) * 128 + htask_q(it) * 8;
        const float4 f0 = __ldcs(reinterpret_cast<const float4 *>(src));
        const float4 f1 = __ldcs(reinterpret_cast<const float4 *>(src + 4));
        const float f[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const __nv_bfloat16 a0 = __float2bfloat16_rn(f[e]), a1 = __float2bfloat16_rn(f[e + 1]);
            hi[e / 2] = bf16_bits(a0) | (bf16_bits(a1) << 16);
            lo[e / 2] = pack_bf16x2(f[e] - __bfloat162float(a0), f[e + 1] - __bfloat162float(a1));
        }
        *reinterpret_cast<uint4 *>(sb + OutLay::kP2 + tck_off(htask_r(it), htask_q(it) * 8)) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        hlo[it] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    // dt and its inclusive prefix sum over the chunk (warps 0..3: warp scans, then the warps' totals in order)
    float dcs = 0.f;
    if (tid < 128) {
        const float d = ld1(dtg + (v * 128 + tid) * a.H + h);
        sdt[tid] = d;
        dcs = d;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, dcs, o);
            if (lane >= o) dcs += u;
        }
        if (lane == 31) wsum[warp] = dcs;
    }
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {  // 256 columns: Yi at 0; G at 128, later Yc
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_addr(&tmem_base))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    __syncthreads();  // wsum
    if (tid < 128) {
        float base = 0.f;
        for (int w = 0; w < warp; ++w) base += wsum[w];
        scs[tid] = base + dcs;
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t taddr = tmem_base;
    const uint32_t base = smem_addr(sb);
    if (tid == 0) {
        for (int kk = 0; kk < 8; ++kk)  // G = C B^T
            tc_mma_i(taddr + 128, tck_desc(base + OutLay::kP0 + kk * 256), tck_desc(base + OutLay::kP1 + kk * 256),
                     kTCIdescKK, kk > 0 ? 1u : 0u);
        for (int kk = 0; kk < 8; ++kk)  // Yi = C H0^T, high part
            tc_mma_i(taddr, tck_desc(base + OutLay::kP0 + kk * 256), tck_desc(base + OutLay::kP2 + kk * 256),
                     kIdescRows, kk > 0 ? 1u : 0u);
        tc_commit(&bar);
    }
    // this thread's 8 x 8 block of x (tokens s0 .. s0+7, rows p0 .. p0+7), loaded while the products run
    // (PR / 8 row blocks x 16 token blocks: threads past them hold none)
    constexpr int kPB = PR / 8;
    const bool hasx = tid < kPB * 16;
    const int bp = tid % kPB, bs = tid / kPB, p0 = bp * 8, s0 = bs * 8;
    uint4 xr[8];
    if (hasx) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            xr[i] = __ldg(reinterpret_cast<const uint4 *>(xg + ((v * 128 + s0 + i) * a.H + h) * (long long)a.P + row0 +
                                                          p0));
    }
    bool ok = mbar_wait_bounded(&bar, 0u);
    int phase = 1;
    if (!__syncthreads_or(!ok)) {
        // B is no longer read: the low part of H0 takes its place; Yi += C H0^T, low part
#pragma unroll
        for (int it = 0; it < PR / 16; ++it)
            *reinterpret_cast<uint4 *>(sb + OutLay::kP1 + tck_off(htask_r(it), htask_q(it) * 8)) = hlo[it];
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            for (int kk = 0; kk < 8; ++kk)
                tc_mma_i(taddr, tck_desc(base + OutLay::kP0 + kk * 256), tck_desc(base + OutLay::kP1 + kk * 256),
                         kIdescRows, 1u);
            tc_commit(&bar);
        }
        ok = mbar_wait_bounded(&bar, 1u);
        phase = 2;
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int t = (warp & 3) * 32 + lane;  // this thread's token (tensor-memory lane)
    const int ch = (warp >> 2) * 64;       // its half of the 128 G columns (and of the PR y columns: ch * PR / 128)
    const uint32_t trow = taddr + ((uint32_t)((warp & 3) * 32) << 16);
    if (__syncthreads_or(!ok)) {
        if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_TIMEOUT);
        mbar_wait_bounded(&bar, (uint32_t)(phase - 1) & 1u);
    } else {
        // every product so far is done: M = mask(G) o decay o dt in two bf16 parts (rows t, K-major) over
        // H0 part 1 and C; x transposed over H0 part 2 (row p, token s)
        const float cst = scs[t];
#pragma unroll 1
        for (int c = ch; c < ch + 64; c += 16) {
            float g[16];
            tc_ld16(trow + 128 + c, g);
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                float m[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int sx = c + e + k;
                    m[k] = sx <= t ? __fmul_rn(__fmul_rn(g[e + k], expf(__fmul_rn(Ah, cst - scs[sx]))), sdt[sx]) : 0.f;
                }
                const __nv_bfloat16 b0 = __float2bfloat16_rn(m[0]), b1 = __float2bfloat16_rn(m[1]);
                hi[e / 2] = bf16_bits(b0) | (bf16_bits(b1) << 16);
                lo[e / 2] = pack_bf16x2(m[0] - __bfloat162float(b0), m[1] - __bfloat162float(b1));
            }
            *reinterpret_cast<uint4 *>(sb + OutLay::kP2 + tck_off(t, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(sb + OutLay::kP2 + tck_off(t, c + 8)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
            *reinterpret_cast<uint4 *>(sb + OutLay::kP0 + tck_off(t, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4 *>(sb + OutLay::kP0 + tck_off(t, c + 8)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        }
        if (hasx) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int j = (k + lane) & 7;  // row p0 + j: element j of each token row; rotated per lane
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) w[e / 2] = u16_at(xr[e], j) | (u16_at(xr[e + 1], j) << 16);
                *reinterpret_cast<uint4 *>(sb + OutLay::kP1 + tck_off(p0 + j, s0)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
        fence_proxy_async_smem();
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();  // every thread is done reading G: Yc may overwrite it
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (tid == 0) {
            for (int kk = 0; kk < 8; ++kk)  // Yc = M X, both parts of M
                tc_mma_i(taddr + 128, tck_desc(base + OutLay::kP2 + kk * 256), tck_desc(base + OutLay::kP1 + kk * 256),
                         kIdescRows, kk > 0 ? 1u : 0u);
            for (int kk = 0; kk < 8; ++kk)
                tc_mma_i(taddr + 128, tck_desc(base + OutLay::kP0 + kk * 256), tck_desc(base + OutLay::kP1 + kk * 256),
                         kIdescRows, 1u);
            tc_commit(&bar);
        }
        // this thread's x values for D x (row t, its half of the columns), from L2 while the product runs
        constexpr int kHalf = PR / 2;  // y columns per thread
        const int cy = (warp >> 2) * kHalf;
        const __nv_bfloat16 *xrow = xg + ((v * 128 + t) * a.H + h) * (long long)a.P + row0 + cy;
        uint4 xd[kHalf / 8];
#pragma unroll
        for (int i = 0; i < kHalf / 8; ++i) xd[i] = __ldg(reinterpret_cast<const uint4 *>(xrow + 8 * i));
        ok = mbar_wait_bounded(&bar, 0u);  // third phase
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (__syncthreads_or(!ok)) {
            if (tid == 0 && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_TIMEOUT);
            mbar_wait_bounded(&bar, 0u);
        } else if (write_y) {
            // y = w_t Yi + Yc + D x, this thread's half of row t, staged through shared memory (over the
            // operands, which the products no longer read) so that each warp writes whole 512-byte rows
            const float wt = expf(__fmul_rn(Ah, cst));
            float *stage = sm<float>(0);  // [128][kStagePitch]
#pragma unroll
            for (int cc = 0; cc < kHalf / 16; ++cc) {
                const int c0 = cy + cc * 16;
                float yi[16], yc[16];
                tc_ld16(trow + c0, yi);
                tc_ld16(trow + 128 + c0, yc);
#pragma unroll
                for (int k = 0; k < 16; k += 4) {
                    float o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int idx = cc * 16 + k + e;
                        const float xv = __uint_as_float(u16_at(xd[idx >> 3], idx & 7) << 16);
                        o[e] = __fmaf_rn(wt, yi[k + e], yc[k + e]) + __fmul_rn(Dh, xv);
                    }
                    *reinterpret_cast<float4 *>(stage + t * kStagePitch + c0 + k) = make_float4(o[0], o[1], o[2], o[3]);
                }
            }
            __syncthreads();  // write_y is the same for the whole CTA
#pragma unroll 4
            for (int it = 0; it < PR / 8; ++it) {  // 128 rows x PR / 4 vectors
                const int idx = it * kOutThreads + tid, row = idx / (PR / 4), c4 = (idx % (PR / 4)) * 4;
                __stcs(reinterpret_cast<float4 *>(a.y + ((v * 128 + row) * a.H + h) * (long long)a.P + row0 + c4),
                       *reinterpret_cast<const float4 *>(stage + row * kStagePitch + c4));
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(taddr) : "memory");
}

// Chunked prefill, the pass between the chunk passes: carry the state across a
// prompt's chunks. Chunk c of sequence b, started from h = 0, left S_c in
// ws[b * nch + c]; with lambda_c the product of its tokens' Abar,
//     H_c = lambda_c H_{c-1} + S_c,   H_{-1} = the sequence's cached state,
// which is the recurrence over the whole prompt regrouped by chunks. Each
// chunk's slot of ws is overwritten with H_{c-1} (the state the chunk starts
// from, for the output pass) and H_{nch-1} goes back to the cache.
struct ScanArgs {
    float *pool;            // cached states [nslots][H][P][N]
    const int32_t *slot;    // pool slot of each sequence (nullptr: slot b)
    int nslots;
    float *ws;              // [batch * nch][H][P][N]
    int32_t *vslot;         // [batch * nch]: chunk c of sequence b -> b * nch + c, or -1 for an invalid slot
    const float *lamw;      // [batch * nch][H]: lambda_c from the first pass, or nullptr: formed here from dt
    const void *dt;         // [batch][T][H]
    int in_bf16;
    const float *A;
    uint32_t *dev_status;
    int H, nch, L;          // heads, chunks, tokens per chunk
    long long PN;           // P * N
};

constexpr int kScanThreads = 256;
constexpr int kScanPerThread = 4;  // state elements per thread: one 16-byte vector
constexpr int kScanAhead = 8;      // chunks whose loads are issued before the carry chain consumes them

__device__ __forceinline__ float4 fma4(float l, float4 h, float4 s) {
    return make_float4(fmaf(l, h.x, s.x), fmaf(l, h.y, s.y), fmaf(l, h.z, s.z), fmaf(l, h.w, s.w));
}

// (launch bounds of two CTAs per SM: the register budget of four spilled the eight chunk vectors in flight)
__global__ void __launch_bounds__(kScanThreads, 2) ssm_chunk_scan_kernel(const ScanArgs a) {
    extern __shared__ float lam[];  // [nch]
    const int b = blockIdx.z, h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float Ah = __ldg(a.A + h);
    int sidx = b;
    bool ok = true;
    if (a.slot != nullptr) {
        sidx = __ldg(a.slot + b);
        ok = sidx >= 0 && sidx < a.nslots;
    }
    // this thread's vector of the cached state and of the first chunks' states: loads issued before the
    // chunk decays are formed, so their latencies overlap
    const long long e = ((long long)blockIdx.x * kScanThreads + tid) * kScanPerThread;  // P * N % 4 == 0
    const bool live = e < a.PN;
    const long long cstride = (long long)a.H * a.PN / kScanPerThread;  // chunk to chunk, in vectors
    float4 *cache = ok && live ? reinterpret_cast<float4 *>(a.pool + ((long long)sidx * a.H + h) * a.PN + e) : nullptr;
    float4 *w = live ? reinterpret_cast<float4 *>(a.ws + ((long long)b * a.nch * a.H + h) * a.PN + e) : nullptr;
    float4 H = make_float4(0.f, 0.f, 0.f, 0.f);  // an invalid slot starts from h = 0
    float4 S[kScanAhead];
    if (live) {
        if (cache != nullptr) H = *cache;
#pragma unroll
        for (int k = 0; k < kScanAhead; ++k)
            if (k < a.nch) S[k] = __ldcs(w + k * cstride);
    }
    // lambda_c: from the first pass where it formed them, else one warp per chunk, a fixed product tree
    // over the chunk's tokens
    if (a.lamw != nullptr) {
        for (int c = tid; c < a.nch; c += kScanThreads) lam[c] = __ldg(a.lamw + ((long long)b * a.nch + c) * a.H + h);
    } else {
        for (int c = warp; c < a.nch; c += kScanThreads / 32) {
            float prod = 1.f;
            for (int i = lane; i < a.L; i += 32) {
                const long long t = (long long)b * a.nch * a.L + (long long)c * a.L + i;
                const float dtv = a.in_bf16 ? ld1(static_cast<const __nv_bfloat16 *>(a.dt) + t * a.H + h)
                                            : ld1(static_cast<const float *>(a.dt) + t * a.H + h);
                prod = __fmul_rn(prod, ssm_decay(dtv, Ah));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) prod = __fmul_rn(prod, __shfl_xor_sync(~0u, prod, off));
            if (lane == 0) lam[c] = prod;
        }
    }
    if (!ok && blockIdx.x == 0 && h == 0 && tid == 0 && a.dev_status != nullptr)
        atomicOr(a.dev_status, SSM_STATUS_BAD_SLOT);
    if (a.vslot != nullptr && blockIdx.x == 0 && h == 0)
        for (int c = tid; c < a.nch; c += kScanThreads) a.vslot[b * a.nch + c] = ok ? b * a.nch + c : -1;
    __syncthreads();
    if (!live) return;
    for (int c0 = 0; c0 < a.nch; c0 += kScanAhead) {
        if (c0 > 0) {
#pragma unroll
            for (int k = 0; k < kScanAhead; ++k)
                if (c0 + k < a.nch) S[k] = __ldcs(w + (c0 + k) * cstride);
        }
#pragma unroll
        for (int k = 0; k < kScanAhead; ++k) {
            if (c0 + k < a.nch) {
                w[(c0 + k) * cstride] = H;
                H = fma4(lam[c0 + k], H, S[k]);
            }
        }
    }
    if (cache != nullptr) *cache = H;
}

// Fixed device scratch of ssm_prefill_scratch: the chunked prefill's
// workspace for callers that do not allocate one. Every call in one CUDA
// context shares it, so calls that may overlap on the device (other streams,
// other host threads, a call still running) race on it.
static __device__ __align__(256) unsigned char g_prefill_scratch[SSM_PREFILL_SCRATCH_BYTES];

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
    if (d->nlayers < 0) return SSM_ERR_SHAPE;
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

int device_sms();

template <typename Tin, int N, int F>
cudaError_t launch_t(const Args &a, cudaStream_t s) {
    constexpr int THREADS = kThreads;
    constexpr int SMEM = Lay<Tin, N, F>::kBytes;
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
    if (grid > device_sms()) {
        kern<<<(unsigned)grid, THREADS, SMEM, s>>>(a);
        return cudaGetLastError();
    }
    // No more CTAs than SMs (a decode step of a few sequences): launched with programmatic dependence on
    // the previous kernel of the stream, so that its launch overlaps that kernel's end; the kernel waits
    // for it before any global access. Plain decode of one Llama-3-8B-shaped layer: 4.63 against 4.77 us.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
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
    bool pool = false;              // `state` is a pool of nslots sequence states
    const int32_t *slot = nullptr;  // pool slot of each sequence (nullptr: slot b for sequence b)
    int nslots = 0;
    bool zero_state = false;        // internal: every tile starts from h = 0, nothing is read
    bool accept_all = false;        // internal: the replay block is replayed in full (no accept_len)
};

// Validate everything on the host, then launch (with dry: validate only).
int run(const ssm_desc_t *d, const Call &c, void *stream, bool dry = false) {
    int rc = check_desc(d);
    if (rc != SSM_OK) return rc;
    const int F = c.flavour;
    const bool verify_phase = F != kCommit;
    const bool replay = F == kCommit || F == kCommitVerify;
    const int rep_K = F == kCommit ? d->ntok : c.rep_ntok;
    if (F == kCommitVerify && rep_K < 1) return SSM_ERR_SHAPE;
    const int N = d->dstate;
    const int ROWS = rows_per_tile(N);
    const int64_t nl = d->nlayers > 1 ? d->nlayers : 1;  // layers; a stack is nl x batch sequences
    const int64_t ptiles = (d->headdim + ROWS - 1) / ROWS;
    const int64_t ntiles = nl * d->batch * d->nheads * ptiles;
    if (ntiles >= (int64_t)1 << 31) return SSM_ERR_SHAPE;
    if (d->batch == 0) return SSM_OK;

    const void *st = F == kVerify ? static_cast<const void *>(c.state_in) : static_cast<const void *>(c.state);
    if ((st == nullptr && !c.zero_state) || c.A == nullptr) return SSM_ERR_NULL;
    if (c.pool) {
        if (c.nslots < 1) return SSM_ERR_SHAPE;
        if (c.slot == nullptr && c.nslots < d->batch) return SSM_ERR_SHAPE;
        if (c.slot != nullptr && !aligned(c.slot, 4)) return SSM_ERR_ALIGN;
    }
    if (verify_phase && (c.x == nullptr || c.B == nullptr || c.C == nullptr || c.dt == nullptr || c.D == nullptr ||
                         c.y == nullptr))
        return SSM_ERR_NULL;
    if (replay && (c.xr == nullptr || c.Br == nullptr || c.dtr == nullptr || (c.accept_len == nullptr && !c.accept_all)))
        return SSM_ERR_NULL;

    const uintptr_t eb = d->in_dtype == SSM_BF16 ? 2 : 4;
    if ((st != nullptr && !aligned(st, 16)) || !aligned(c.A, 4)) return SSM_ERR_ALIGN;
    if (verify_phase && (!aligned(c.x, eb) || !aligned(c.B, eb) || !aligned(c.C, eb) || !aligned(c.dt, eb) ||
                         !aligned(c.D, 4) || !aligned(c.y, 4)))
        return SSM_ERR_ALIGN;
    if (replay && (!aligned(c.xr, eb) || !aligned(c.Br, eb) || !aligned(c.dtr, eb))) return SSM_ERR_ALIGN;
    if (c.accept_len != nullptr && !aligned(c.accept_len, 4)) return SSM_ERR_ALIGN;
    if (c.dev_status != nullptr && !aligned(c.dev_status, 4)) return SSM_ERR_ALIGN;

    // B_: sequences of the call (all layers); accept_len covers one layer's d->batch
    const int64_t B_ = nl * d->batch, H = d->nheads, P = d->headdim, G = d->ngroups;
    const int64_t state_bytes = (c.pool ? nl * c.nslots : B_) * H * P * N * 4;
    BufList bl;
    if (st != nullptr) bl.add(st, state_bytes, F != kVerify);
    if (c.pool && c.slot != nullptr) bl.add(c.slot, (int64_t)d->batch * 4, false);
    bl.add(c.A, nl * H * 4, false);
    if (verify_phase) {
        const int64_t bk = B_ * d->ntok;
        bl.add(c.x, bk * H * P * eb, false);
        bl.add(c.B, bk * G * N * eb, false);
        bl.add(c.C, bk * G * N * eb, false);
        bl.add(c.dt, bk * H * eb, false);
        bl.add(c.D, nl * H * 4, false);
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
    if (c.accept_len != nullptr) bl.add(c.accept_len, (int64_t)d->batch * 4, false);
    if (c.dev_status != nullptr) bl.add(c.dev_status, 4, true);
    if (!bl.disjoint_writes()) return SSM_ERR_ALIAS;
    if (dry) return SSM_OK;

    Args a;
    a.state_in = c.zero_state ? nullptr : static_cast<const float *>(st);
    a.state = F == kVerify ? nullptr : c.state;
    a.slot = c.pool ? c.slot : nullptr;
    a.nslots = c.pool ? c.nslots : 0;
    const uintptr_t rowb = (uintptr_t)P * eb;
    a.ver.x = c.x;
    a.ver.B = c.B;
    a.ver.C = c.C;
    a.ver.dt = c.dt;
    a.ver.K = d->ntok;
    a.ver.vec_x = verify_phase && aligned(c.x, 16) && rowb % 16 == 0;
    a.ver.vec_bc = verify_phase && aligned(c.B, 16) && aligned(c.C, 16);
    a.ver.tma = a.ver.vec_x && a.ver.vec_bc;
    a.rep.x = c.xr;
    a.rep.B = c.Br;
    a.rep.C = nullptr;
    a.rep.dt = c.dtr;
    a.rep.K = rep_K;
    a.rep.vec_x = replay && aligned(c.xr, 16) && rowb % 16 == 0;
    a.rep.vec_bc = replay && aligned(c.Br, 16);
    a.rep.tma = a.rep.vec_x && a.rep.vec_bc;
    a.A = c.A;
    a.D = c.D;
    a.accept_len = c.accept_len;
    a.y = c.y;
    a.dev_status = c.dev_status;
    a.H = d->nheads;
    a.P = d->headdim;
    a.G = d->ngroups;
    a.ptiles = (int)ptiles;
    a.bpl = d->batch;
    a.fd_ptiles = make_fdiv((uint32_t)ptiles);
    a.fd_H = make_fdiv((uint32_t)d->nheads);
    a.fd_bpl = make_fdiv((uint32_t)d->batch);
    a.fd_hpg = make_fdiv((uint32_t)(d->nheads / d->ngroups));
    a.ntiles = ntiles;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    const int FX = F | (c.pool ? kPoolBit : 0) | (c.zero_state ? kZeroBit : 0);
    switch (FX) {
        case kVerify: e = launch_flavour<kVerify>(d->in_dtype, N, a, s); break;
        case kCommit: e = launch_flavour<kCommit>(d->in_dtype, N, a, s); break;
        case kCommitVerify: e = launch_flavour<kCommitVerify>(d->in_dtype, N, a, s); break;
        case kVerifyCommit: e = launch_flavour<kVerifyCommit>(d->in_dtype, N, a, s); break;
        case kVerify | kPoolBit: e = launch_flavour<kVerify | kPoolBit>(d->in_dtype, N, a, s); break;
        case kCommit | kPoolBit: e = launch_flavour<kCommit | kPoolBit>(d->in_dtype, N, a, s); break;
        case kCommitVerify | kPoolBit: e = launch_flavour<kCommitVerify | kPoolBit>(d->in_dtype, N, a, s); break;
        case kVerifyCommit | kPoolBit: e = launch_flavour<kVerifyCommit | kPoolBit>(d->in_dtype, N, a, s); break;
        case kCommit | kZeroBit: e = launch_flavour<kCommit | kZeroBit>(d->in_dtype, N, a, s); break;
        default: return SSM_ERR_UNSUPPORTED;  // no kernel for this combination
    }
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return SSM_ERR_CUDA;
    }
    return SSM_OK;
}


// SM count of the current device (immutable; cached per device).
int device_sms() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int v = (dev >= 0 && dev < kMaxDevices) ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        if (dev >= 0 && dev < kMaxDevices) cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

constexpr int kMaxChunks = 4096;

// Workspace of a chunked prefill with chunk length L: the chunk states, then
// the chunks' slot map, then each chunk's lambda per head (each part 16-byte
// aligned).
int64_t prefill_ws_states(const ssm_desc_t *d, int L) {
    return (int64_t)d->batch * (d->ntok / L) * d->nheads * d->headdim * d->dstate * 4;
}
int64_t prefill_ws_lam(const ssm_desc_t *d, int L) {
    return prefill_ws_states(d, L) + ((int64_t)d->batch * (d->ntok / L) * 4 + 15) / 16 * 16;
}
int64_t prefill_ws_bytes(const ssm_desc_t *d, int L) {
    return prefill_ws_lam(d, L) + ((int64_t)d->batch * (d->ntok / L) * d->nheads * 4 + 15) / 16 * 16;
}

// Chunk length of a chunked prefill: 128 for the shapes of the tensor-memory
// chunk passes when the workspace holds it; otherwise the largest of 128,
// 64, 32, 16 that divides the prompt into at least two chunks, fits the
// workspace and gives one wave of tiles (four per SM), the smallest fitting
// one if none reaches a wave. 0: the one-pass form (it fills the device by
// itself, or no chunk length fits).
int prefill_chunk_len(const ssm_desc_t *d, int64_t ws_bytes) {
    const int T = d->ntok;
    // shapes the tensor-memory chunk passes take: 128-token chunks whenever the workspace allows, since
    // those passes cost far less per token than the recurrence, whatever the grid
    if (d->in_dtype == SSM_BF16 && d->dstate == 128 && d->headdim % 64 == 0 && T % 128 == 0 && T / 128 >= 2 &&
        T / 128 <= kMaxChunks && (ws_bytes < 0 || prefill_ws_bytes(d, 128) <= ws_bytes))
        return 128;
    const int ROWS = rows_per_tile(d->dstate);
    const int64_t ptiles = (d->headdim + ROWS - 1) / ROWS;
    const int64_t base = (int64_t)d->batch * d->nheads * ptiles;
    const int64_t wave = (int64_t)device_sms() * 4;
    if (wave <= 0 || base >= wave) return 0;
    int best = 0;
    for (int L = kCSMaxL; L >= 16; L >>= 1) {
        if (T % L != 0 || T / L < 2 || T / L > kMaxChunks) continue;
        if (ws_bytes >= 0 && prefill_ws_bytes(d, L) > ws_bytes) continue;
        best = L;
        if (base * (T / L) >= wave) break;
    }
    return best;
}

template <typename Tin, int N>
cudaError_t launch_cs_t(const CSArgs &a, long long ntiles, cudaStream_t s) {
    constexpr int SMEM = CSLay<Tin, N>::kBytes;
    static std::atomic<int> ready[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || ready[dev].load(std::memory_order_relaxed) == 0) {
        e = cudaFuncSetAttribute(ssm_chunk_state_kernel<Tin, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) ready[dev].store(1, std::memory_order_relaxed);
    }
    ssm_chunk_state_kernel<Tin, N><<<(unsigned)ntiles, 128, SMEM, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_chunk_state_tc(const CSArgs &a, long long ntiles, cudaStream_t s) {
    static std::atomic<int> ready[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || ready[dev].load(std::memory_order_relaxed) == 0) {
        e = cudaFuncSetAttribute(ssm_chunk_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TCLay::kBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) ready[dev].store(1, std::memory_order_relaxed);
    }
    ssm_chunk_state_tc_kernel<<<(unsigned)ntiles, kTCThreads, TCLay::kBytes, s>>>(a);
    return cudaGetLastError();
}

template <int PR>
cudaError_t launch_chunk_out_tc(const OutArgs &a, long long ntiles, cudaStream_t s) {
    static std::atomic<int> ready[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices || ready[dev].load(std::memory_order_relaxed) == 0) {
        e = cudaFuncSetAttribute(ssm_chunk_out_tc_kernel<PR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 OutLay::kBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < kMaxDevices) ready[dev].store(1, std::memory_order_relaxed);
    }
    ssm_chunk_out_tc_kernel<PR><<<(unsigned)ntiles, kOutThreads, OutLay::kBytes, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_chunk_state(int in_dtype, int N, const CSArgs &a, long long ntiles, cudaStream_t s) {
    if (in_dtype == SSM_BF16) {
        switch (N) {
            case 16: return launch_cs_t<__nv_bfloat16, 16>(a, ntiles, s);
            case 32: return launch_cs_t<__nv_bfloat16, 32>(a, ntiles, s);
            case 64: return launch_cs_t<__nv_bfloat16, 64>(a, ntiles, s);
            default: return launch_cs_t<__nv_bfloat16, 128>(a, ntiles, s);
        }
    }
    switch (N) {
        case 16: return launch_cs_t<float, 16>(a, ntiles, s);
        case 32: return launch_cs_t<float, 32>(a, ntiles, s);
        case 64: return launch_cs_t<float, 64>(a, ntiles, s);
        default: return launch_cs_t<float, 128>(a, ntiles, s);
    }
}

int prefill(const ssm_desc_t *d, const ssm_pool_t *pool, const void *x, const void *B, const void *C,
            const void *dt, const float *A, const float *D, float *y, void *ws, int64_t ws_bytes,
            uint32_t *dev_status, void *stream) {
    int rc = check_desc(d);
    if (rc != SSM_OK) return rc;
    if (d->nlayers > 1) return SSM_ERR_UNSUPPORTED;  // one layer per prefill
    if (pool == nullptr) return SSM_ERR_NULL;
    if (pool->reserved != 0 || ws_bytes < 0) return SSM_ERR_SHAPE;
    if (d->batch == 0) return SSM_OK;
    Call c{};
    c.flavour = kVerifyCommit;  // every prompt token is kept: accept_len = nullptr means all
    c.state = pool->states;
    c.pool = true;
    c.slot = pool->slot;
    c.nslots = pool->nslots;
    c.x = x; c.B = B; c.C = C; c.dt = dt;
    c.A = A; c.D = D; c.y = y;
    c.dev_status = dev_status;
    rc = run(d, c, stream, true);
    if (rc != SSM_OK) return rc;
    const int L = prefill_chunk_len(d, ws == nullptr ? 0 : ws_bytes);
    if (L == 0) return run(d, c, stream);

    // Chunked: (1) every chunk from h = 0 -> ws; (2) carry across chunks;
    // (3) y of every chunk from the state it starts from.
    const int nch = d->ntok / L;
    const int64_t H = d->nheads, P = d->headdim, N = d->dstate, G = d->ngroups, Bn = d->batch;
    const int64_t need = prefill_ws_bytes(d, L);
    if (!aligned(ws, 16)) return SSM_ERR_ALIGN;
    const uintptr_t eb = d->in_dtype == SSM_BF16 ? 2 : 4;
    const int64_t bt = Bn * d->ntok;
    const Range w = range_of(ws, need);
    const Range others[] = {range_of(pool->states, (int64_t)pool->nslots * H * P * N * 4),
                            range_of(x, bt * H * P * eb), range_of(B, bt * G * N * eb), range_of(C, bt * G * N * eb),
                            range_of(dt, bt * H * eb), range_of(A, H * 4), range_of(D, H * 4),
                            range_of(y, bt * H * P * 4)};
    for (const Range &o : others)
        if (overlaps(w, o)) return SSM_ERR_ALIAS;
    if (pool->slot != nullptr && overlaps(w, range_of(pool->slot, Bn * 4))) return SSM_ERR_ALIAS;
    if (dev_status != nullptr && overlaps(w, range_of(dev_status, 4))) return SSM_ERR_ALIAS;

    ssm_desc_t dv = *d;  // chunk c of sequence b is virtual sequence b * nch + c
    dv.batch = (int32_t)(Bn * nch);
    dv.ntok = L;
    Call c1{};
    c1.flavour = kCommit;
    c1.state = static_cast<float *>(ws);
    c1.zero_state = true;
    c1.accept_all = true;
    c1.xr = x; c1.Br = B; c1.dtr = dt;
    c1.A = A;
    c1.dev_status = dev_status;
    const bool cs_ok = N <= 128 && P % kCSRows == 0 && aligned(x, 16) && aligned(B, 16) && (P * eb) % 16 == 0 &&
                       aligned(dt, eb);
    // the tensor-memory form: bf16 inputs, N = 128, L = 128, tiles of 128 rows of one head, or of two heads of
    // one group at P = 64
    const bool tc_states = cs_ok && d->in_dtype == SSM_BF16 && N == 128 && L == 128 &&
                       (P % kTCRows == 0 || (P == 64 && (H / G) % 2 == 0));
    if (cs_ok) {
        CSArgs ca;
        ca.x = x;
        ca.B = B;
        ca.dt = dt;
        ca.A = A;
        ca.ws = static_cast<float *>(ws);
        ca.lam = reinterpret_cast<float *>(static_cast<char *>(ws) + prefill_ws_lam(d, L));
        ca.dev_status = dev_status;
        ca.H = (int)H;
        ca.P = (int)P;
        ca.G = (int)G;
        ca.L = L;
        // tiles of a chunk: P / 64 per head, or H P / 128 over the chunk's rows on the tensor cores
        ca.ptiles = tc_states ? (int)(H * P / kTCRows) : (int)(P / kCSRows);
        const long long nt = (long long)dv.batch * (tc_states ? ca.ptiles : H * ca.ptiles);
        const cudaError_t e1 = tc_states ? launch_chunk_state_tc(ca, nt, static_cast<cudaStream_t>(stream))
                                     : launch_chunk_state(d->in_dtype, (int)N, ca, nt, static_cast<cudaStream_t>(stream));
        if (e1 != cudaSuccess) {
            g_last_cuda_error = (int)e1;
            return SSM_ERR_CUDA;
        }
    } else {
        rc = run(&dv, c1, stream);
        if (rc != SSM_OK) return rc;
    }

    ScanArgs sa;
    sa.pool = pool->states;
    sa.slot = pool->slot;
    sa.nslots = pool->nslots;
    sa.ws = static_cast<float *>(ws);
    int32_t *vslot = pool->slot != nullptr
                         ? reinterpret_cast<int32_t *>(static_cast<char *>(ws) + prefill_ws_states(d, L))
                         : nullptr;
    sa.vslot = vslot;
    sa.lamw = cs_ok ? reinterpret_cast<const float *>(static_cast<const char *>(ws) + prefill_ws_lam(d, L)) : nullptr;
    sa.dt = dt;
    sa.in_bf16 = d->in_dtype == SSM_BF16;
    sa.A = A;
    sa.dev_status = dev_status;
    sa.H = (int)H;
    sa.nch = nch;
    sa.L = L;
    sa.PN = P * N;
    const dim3 grid((unsigned)((P * N / kScanPerThread + kScanThreads - 1) / kScanThreads),
                    (unsigned)H, (unsigned)Bn);
    ssm_chunk_scan_kernel<<<grid, kScanThreads, nch * sizeof(float), static_cast<cudaStream_t>(stream)>>>(sa);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return SSM_ERR_CUDA;
    }

    // the chunked output form on the tensor cores: bf16, N = 128, 128-token chunks, 64- or 128-row tiles
    const bool tc_out = cs_ok && d->in_dtype == SSM_BF16 && N == 128 && L == 128 && P % 64 == 0 && aligned(C, 16) &&
                        aligned(y, 16);
    if (tc_out) {
        OutArgs oa;
        oa.x = x; oa.B = B; oa.C = C; oa.dt = dt;
        oa.A = A; oa.D = D;
        oa.ws = static_cast<const float *>(ws);
        oa.vslot = vslot;
        oa.y = y;
        oa.dev_status = dev_status;
        oa.H = (int)H; oa.P = (int)P; oa.G = (int)G;
        const int pr = P % 128 == 0 ? 128 : 64;
        oa.ptiles = (int)(P / pr);
        const long long nt3 = (long long)dv.batch * H * (P / pr);
        const cudaError_t e3 = pr == 128 ? launch_chunk_out_tc<128>(oa, nt3, static_cast<cudaStream_t>(stream))
                                         : launch_chunk_out_tc<64>(oa, nt3, static_cast<cudaStream_t>(stream));
        if (e3 != cudaSuccess) {
            g_last_cuda_error = (int)e3;
            return SSM_ERR_CUDA;
        }
        return SSM_OK;
    }
    Call c3{};
    c3.flavour = kVerify;
    c3.state_in = static_cast<const float *>(ws);
    if (vslot != nullptr) {  // chunks of sequences without a valid slot write no y
        c3.pool = true;
        c3.slot = vslot;
        c3.nslots = dv.batch;
    }
    c3.x = x; c3.B = B; c3.C = C; c3.dt = dt;
    c3.A = A; c3.D = D; c3.y = y;
    c3.dev_status = dev_status;
    return run(&dv, c3, stream);
}

// Device address of the prefill scratch in the current context. It is looked
// up on every call, not cached: after cudaDeviceReset, or in another context
// on the same device, the library's device code is loaded again and the array
// may sit elsewhere, so a remembered address could point at unmapped or
// foreign memory. The lookup is cheap next to the kernels it feeds.
void *prefill_scratch(cudaError_t &err) {
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_prefill_scratch);
    return err == cudaSuccess ? p : nullptr;
}

Call pool_call(int flavour, const ssm_pool_t *pool) {
    Call c{};
    c.flavour = flavour;
    c.pool = true;
    if (pool != nullptr) {
        c.state = pool->states;
        c.state_in = pool->states;
        c.slot = pool->slot;
        c.nslots = pool->nslots;
    }
    return c;
}

int check_pool(const ssm_pool_t *pool) {
    if (pool == nullptr) return SSM_ERR_NULL;
    if (pool->reserved != 0) return SSM_ERR_SHAPE;
    return SSM_OK;
}

}  // namespace

namespace ssm_internal {
void set_last_cuda_error(int e) { g_last_cuda_error = e; }
}  // namespace ssm_internal

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

int ssm_verify_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *C,
                    const void *dt, const float *A, const float *D, float *y, uint32_t *dev_status, void *stream) {
    const int rc = check_pool(pool);
    if (rc != SSM_OK) return rc;
    Call c = pool_call(kVerify, pool);
    c.x = x; c.B = B; c.C = C; c.dt = dt;
    c.A = A; c.D = D; c.y = y;
    c.dev_status = dev_status;
    return run(desc, c, stream);
}

int ssm_commit_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *dt,
                    const float *A, const int32_t *accept_len, uint32_t *dev_status, void *stream) {
    const int rc = check_pool(pool);
    if (rc != SSM_OK) return rc;
    Call c = pool_call(kCommit, pool);
    c.xr = x; c.Br = B; c.dtr = dt;
    c.A = A;
    c.accept_len = accept_len;
    c.dev_status = dev_status;
    return run(desc, c, stream);
}

int ssm_verify_commit_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B,
                           const void *C, const void *dt, const float *A, const float *D, const int32_t *accept_len,
                           float *y, uint32_t *dev_status, void *stream) {
    const int rc = check_pool(pool);
    if (rc != SSM_OK) return rc;
    if (accept_len == nullptr && desc != nullptr && desc->batch > 0) return SSM_ERR_NULL;
    Call c = pool_call(kVerifyCommit, pool);
    c.x = x; c.B = B; c.C = C; c.dt = dt;
    c.A = A; c.D = D; c.y = y;
    c.accept_len = accept_len;
    c.dev_status = dev_status;
    return run(desc, c, stream);
}

int ssm_commit_verify_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, int32_t prev_ntok, const void *x_prev,
                           const void *B_prev, const void *dt_prev, const int32_t *accept_len_prev, const void *x,
                           const void *B, const void *C, const void *dt, const float *A, const float *D, float *y,
                           uint32_t *dev_status, void *stream) {
    const int rc = check_pool(pool);
    if (rc != SSM_OK) return rc;
    Call c = pool_call(kCommitVerify, pool);
    c.rep_ntok = prev_ntok;
    c.xr = x_prev; c.Br = B_prev; c.dtr = dt_prev;
    c.accept_len = accept_len_prev;
    c.x = x; c.B = B; c.C = C; c.dt = dt;
    c.A = A; c.D = D; c.y = y;
    c.dev_status = dev_status;
    return run(desc, c, stream);
}

int ssm_step_pool(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *C,
                  const void *dt, const float *A, const float *D, float *y, uint32_t *dev_status, void *stream) {
    const int rc = check_pool(pool);
    if (rc != SSM_OK) return rc;
    if (desc != nullptr && desc->ntok != 1) return SSM_ERR_SHAPE;
    Call c = pool_call(kVerifyCommit, pool);
    c.x = x; c.B = B; c.C = C; c.dt = dt;
    c.A = A; c.D = D; c.y = y;
    c.dev_status = dev_status;
    return run(desc, c, stream);
}

int64_t ssm_prefill_workspace_bytes(const ssm_desc_t *desc) {
    if (check_desc(desc) != SSM_OK || desc->batch == 0 || desc->nlayers > 1) return 0;
    const int L = prefill_chunk_len(desc, -1);
    return L == 0 ? 0 : prefill_ws_bytes(desc, L);
}

int ssm_prefill(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *C,
                const void *dt, const float *A, const float *D, float *y, void *workspace, int64_t workspace_bytes,
                uint32_t *dev_status, void *stream) {
    return prefill(desc, pool, x, B, C, dt, A, D, y, workspace, workspace_bytes, dev_status, stream);
}

int ssm_prefill_scratch(const ssm_desc_t *desc, const ssm_pool_t *pool, const void *x, const void *B, const void *C,
                        const void *dt, const float *A, const float *D, float *y, uint32_t *dev_status, void *stream) {
    const int rc = check_desc(desc);
    if (rc != SSM_OK) return rc;
    if (desc->nlayers > 1) return SSM_ERR_UNSUPPORTED;
    if (pool == nullptr) return SSM_ERR_NULL;
    if (desc->batch == 0) return SSM_OK;
    // the chunk length the fixed scratch holds (0: the one-pass form, which needs no workspace)
    const int L = prefill_chunk_len(desc, SSM_PREFILL_SCRATCH_BYTES);
    const int64_t need = L > 0 ? prefill_ws_bytes(desc, L) : 0;
    void *ws = nullptr;
    if (need > 0) {
        cudaError_t e = cudaSuccess;
        ws = prefill_scratch(e);
        if (ws == nullptr) {
            g_last_cuda_error = (int)e;
            return SSM_ERR_CUDA;
        }
    }
    return prefill(desc, pool, x, B, C, dt, A, D, y, ws, need, dev_status, stream);
}

int ssm_selftest_wait_timeout(uint32_t *dev_status, void *stream) {
    if (dev_status == nullptr) return SSM_ERR_NULL;
    if (!aligned(dev_status, 4)) return SSM_ERR_ALIGN;
    ssm_wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        g_last_cuda_error = (int)e;
        return SSM_ERR_CUDA;
    }
    return SSM_OK;
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
