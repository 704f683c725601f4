// libssmverify: acceptance of draft tokens on the device (sm_103a).
//
// The step right after the verifier's pass in speculative decoding: news
// summary "Llama 3+Mamba强强联手！蒸馏到RNN，推理速度提升1.6倍",
// speculative-decoding section (the draft proposes K tokens; tokens the
// verifier agrees with are accepted; at the first one it does not, the rest
// are dropped and the state rolls back to the last accepted token; with all K
// accepted the next round starts), with the method overview naming it a
// speculative sampling algorithm. Two rules, per sequence b:
//   greedy:   accept draft token t while it is the verifier's most likely
//             token at t; next token = the verifier's most likely token at
//             j = accept_len (ties to the smallest index).
//   sampling: p_t = softmax(target logits t), q_t = softmax(draft logits t);
//             accept x_t while u_t < p_t(x_t) / q_t(x_t); next token = the
//             inverse CDF at u_K of max(0, p_j - q_j) (j < K) or of p_K.
// accept_len lands in device memory, ready for ssm_commit /
// ssm_commit_verify without a trip through the host.
//
// Kernel design (B300; bound by the HBM stream of the logits it must read):
//  * One thread-block cluster of kCl CTAs per sequence; CTA r owns a slice
//    of V / kCl vocabulary entries of each row it reads and streams it with 16-byte
//    loads, kAU of them in flight per thread.
//  * The rule only ever looks at rows up to the first rejection, so the
//    rows are read in steps of kGroup draft tokens (their verifier rows and,
//    for sampling, their draft rows) and the walk stops at the step holding
//    the first rejection: rows past it are never read. (One token per step
//    exposes a load latency and a cluster barrier per token; three per step
//    measured fastest.)
//  * Per row, each thread keeps a running (max, sum of exp(l - max)) -- the
//    online softmax normaliser -- or a running (max, first index of the
//    max); warps, then the CTA, then the cluster combine these partials. The
//    cluster step reads every CTA's partials through distributed shared
//    memory in rank order, so every CTA of the cluster holds bit-identical
//    row statistics and takes the same decisions without further exchange.
//    The partials of consecutive steps alternate between two buffers, so one
//    cluster barrier per step suffices.
//  * Sampling then draws the next token: every CTA sums the weights of its
//    slice of row j (each thread a contiguous run, a block prefix over
//    threads, a cluster prefix over CTAs); the CTA and thread whose range
//    holds the threshold rescan that run. The search uses the same rounded
//    partial sums at every level, so it always ends on an index of positive
//    weight.
//  * exp(l - m) is taken as 2^(l log2 e - m log2 e) with the hardware's base-2
//    exponential (PTX ex2.approx, relative error about 2^-22, subnormal
//    results flushed to zero): the change of base used by fused softmax
//    kernels such as FlashAttention. Probabilities are fp32; sums are fp32.

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cooperative_groups.h>

#include <climits>
#include <type_traits>
#include <stdint.h>

#include "ssmverify.h"
#include "ssm_internal.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kAT = 256;                             // threads per CTA
constexpr int kAWarps = kAT / 32;
constexpr int kAU = 8;                               // 16-byte loads in flight per thread and batch
constexpr int kAS = 16;                              // elements per thread and batch on the scalar path
constexpr int kCl = 8;                               // CTAs per sequence (one cluster)
constexpr int kGroup = 3;                            // draft tokens whose rows are read and decided per step
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kEmpty = -1.0e30f;                   // running max of a partial that has seen nothing
constexpr int kNoIndex = INT_MAX;

struct AArgs {
    const void *tl;          // verifier logits [batch][K + 1][V]
    const void *ql;          // draft logits [batch][K][V] (sampling only)
    const int32_t *drafts;   // [batch][K]
    const float *u;          // [batch][K + 1] (sampling only)
    int32_t *accept_len;     // [batch]
    int32_t *next_token;     // [batch]
    uint32_t *dev_status;    // nullable
    int K, V;
    int slice;               // vocabulary entries per CTA (a multiple of the vector width)
};

// 2^x, PTX ex2.approx with subnormal results flushed to zero.
__device__ __forceinline__ float exp2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16-byte load that bypasses L1 (the logits are streamed once).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t word(const uint4 &r, int i) {
    return i == 0 ? r.x : i == 1 ? r.y : i == 2 ? r.z : r.w;
}

template <typename T>
struct Logit;

template <>
struct Logit<float> {
    static constexpr int W = 4;                          // per 16-byte vector
    static constexpr uint32_t kNegInf = 0xff800000u;     // one -inf per word
    __device__ static float get(const uint4 &r, int l) { return __uint_as_float(word(r, l)); }
    __device__ static float one(const float *p) { return __ldg(p); }
    __device__ static float2 pair(const uint4 &r, int q) {  // elements 2q, 2q + 1
        return q == 0 ? make_float2(__uint_as_float(r.x), __uint_as_float(r.y))
                      : make_float2(__uint_as_float(r.z), __uint_as_float(r.w));
    }
    template <int S>
    __device__ static float bmax(const uint4 (&r)[S]) {
        float m0 = fmaxf(get(r[0], 0), get(r[0], 1)), m1 = fmaxf(get(r[0], 2), get(r[0], 3));
#pragma unroll
        for (int k = 1; k < S; ++k) {
            m0 = fmaxf(m0, fmaxf(get(r[k], 0), get(r[k], 1)));
            m1 = fmaxf(m1, fmaxf(get(r[k], 2), get(r[k], 3)));
        }
        return fmaxf(m0, m1);
    }
};

template <>
struct Logit<__nv_bfloat16> {
    static constexpr int W = 8;
    static constexpr uint32_t kNegInf = 0xff80ff80u;     // two bf16 -inf per word
    __device__ static float get(const uint4 &r, int l) {
        const uint32_t w = word(r, l >> 1);
        return __uint_as_float((l & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    __device__ static float one(const __nv_bfloat16 *p) {
        return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(p))) << 16);
    }
    __device__ static uint32_t max2(uint32_t a, uint32_t b) {  // packed bf16x2 max
        __nv_bfloat162 x, y;
        __builtin_memcpy(&x, &a, 4);
        __builtin_memcpy(&y, &b, 4);
        const __nv_bfloat162 m = __hmax2(x, y);
        uint32_t r;
        __builtin_memcpy(&r, &m, 4);
        return r;
    }
    __device__ static float2 pair(const uint4 &r, int q) {  // elements 2q, 2q + 1
        const uint32_t w = word(r, q);
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    template <int S>
    __device__ static float bmax(const uint4 (&r)[S]) {  // packed bf16x2 maxima, unpacked once
        uint32_t m0 = max2(r[0].x, r[0].y), m1 = max2(r[0].z, r[0].w);
#pragma unroll
        for (int k = 1; k < S; ++k) {
            m0 = max2(m0, max2(r[k].x, r[k].y));
            m1 = max2(m1, max2(r[k].z, r[k].w));
        }
        const uint32_t m = max2(m0, m1);
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
    }
};

// A batch of logits of one row seen by one thread, in increasing index order
// (slot k, element l). Masked-out entries read -inf; valid slots come first,
// and a batch whose slot 0 is masked (any == false) holds nothing.
template <typename T, bool VEC>
struct Batch;

template <typename T>
struct Batch<T, true> {
    static constexpr int S = kAU, W = Logit<T>::W;
    static constexpr bool kPaired = true;
    uint4 r[S];
    int v0;     // vector index of slot 0
    bool any;   // slot 0 (and so the batch) holds data
    __device__ void load(const T *row, int v0_, int vhi) {
        v0 = v0_;
        any = v0 < vhi;
        const uint4 *p = reinterpret_cast<const uint4 *>(row);
        if (v0 + (S - 1) * kAT < vhi) {  // the usual case: every slot inside the slice
#pragma unroll
            for (int k = 0; k < S; ++k) r[k] = ld_stream(p + v0 + k * kAT);
        } else {
            const uint4 neg = make_uint4(Logit<T>::kNegInf, Logit<T>::kNegInf, Logit<T>::kNegInf, Logit<T>::kNegInf);
#pragma unroll
            for (int k = 0; k < S; ++k) {
                const int v = v0 + k * kAT;
                r[k] = v < vhi ? ld_stream(p + v) : neg;
            }
        }
    }
    __device__ float get(int k, int l) const { return Logit<T>::get(r[k], l); }
    __device__ float2 pair(int k, int q) const { return Logit<T>::pair(r[k], q); }
    __device__ int index(int k, int l) const { return (v0 + k * kAT) * W + l; }
    __device__ float bmax() const { return Logit<T>::template bmax<S>(r); }
};

template <typename T>
struct Batch<T, false> {
    static constexpr int S = kAS, W = 1;
    static constexpr bool kPaired = false;
    float r[S];
    int e0;
    bool any;
    __device__ void load(const T *row, int e0_, int ehi) {
        e0 = e0_;
        any = e0 < ehi;
#pragma unroll
        for (int k = 0; k < S; ++k) {
            const int e = e0 + k * kAT;
            r[k] = e < ehi ? Logit<T>::one(row + e) : -INFINITY;
        }
    }
    __device__ float get(int k, int) const { return r[k]; }
    __device__ float2 pair(int, int) const { return make_float2(0.f, 0.f); }  // not used (kPaired is false)
    __device__ int index(int k, int) const { return e0 + k * kAT; }
    __device__ float bmax() const {
        float m = r[0];
#pragma unroll
        for (int k = 1; k < S; ++k) m = fmaxf(m, r[k]);
        return m;
    }
};

// Running softmax normaliser: max m and s = sum of exp(l - m).
struct SoftAcc {
    float m = kEmpty, s = 0.f;
    template <class B>
    __device__ void push(const B &b) {
        if (!b.any) return;
        const float bm = b.bmax();
        if (bm > m) {
            s *= exp2_ftz((m - bm) * kLog2e);
            m = bm;
        }
        const float nml = -(m * kLog2e);
        if constexpr (B::kPaired) {
            // two entries per instruction for the exponent argument and the sum
            const float2 l2 = make_float2(kLog2e, kLog2e), n2 = make_float2(nml, nml);
            float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
            for (int k = 0; k < B::S; ++k) {
#pragma unroll
                for (int q = 0; q < B::W / 2; ++q) {
                    const float2 x = __ffma2_rn(b.pair(k, q), l2, n2);
                    const float2 e = make_float2(exp2_ftz(x.x), exp2_ftz(x.y));
                    if ((k * (B::W / 2) + q) & 1)
                        a1 = __fadd2_rn(a1, e);
                    else
                        a0 = __fadd2_rn(a0, e);
                }
            }
            s += (a0.x + a1.x) + (a0.y + a1.y);
        } else {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll
            for (int k = 0; k < B::S; ++k) {
                const float e = exp2_ftz(fmaf(b.get(k, 0), kLog2e, nml));
                if (k & 1)
                    a1 += e;
                else
                    a0 += e;
            }
            s += a0 + a1;
        }
    }
    __device__ float2 warp_total();
};

__device__ __forceinline__ void soft_combine(float &m, float &s, float m2, float s2) {
    const float M = fmaxf(m, m2);
    s = s * exp2_ftz((m - M) * kLog2e) + s2 * exp2_ftz((m2 - M) * kLog2e);
    m = M;
}

__device__ __forceinline__ float2 SoftAcc::warp_total() {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        soft_combine(m, s, __shfl_xor_sync(~0u, m, off), __shfl_xor_sync(~0u, s, off));
    return make_float2(m, s);
}

// Running argmax: the largest value and the smallest index holding it.
struct ArgAcc {
    float v = -INFINITY;
    int i = kNoIndex;
    template <class B>
    __device__ void push(const B &b) {
        if (!b.any) return;
        const float bm = b.bmax();
        if (bm > v || (i == kNoIndex && bm == v)) {
            int idx = kNoIndex;
#pragma unroll
            for (int k = B::S - 1; k >= 0; --k) {
#pragma unroll
                for (int l = B::W - 1; l >= 0; --l)
                    if (b.get(k, l) == bm) idx = b.index(k, l);
            }
            v = bm;
            i = idx;
        }
    }
    __device__ float2 warp_total();
};

__device__ __forceinline__ void arg_combine(float &v, int &i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

__device__ __forceinline__ float2 ArgAcc::warp_total() {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        arg_combine(v, i, __shfl_xor_sync(~0u, v, off), __shfl_xor_sync(~0u, i, off));
    return make_float2(v, __int_as_float(i));
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// The weight of one vocabulary entry for the next-token draw: p (= e / S of
// the verifier row) or max(0, p - q). Explicit roundings, so that every
// evaluation of the same entry gives the same bits.
struct Weigher {
    bool resid;
    float nmlp, invp, nmlq, invq;
    __device__ float operator()(float lp, float lq) const {
        const float p = __fmul_rn(exp2_ftz(fmaf(lp, kLog2e, nmlp)), invp);
        if (!resid) return p;
        const float q = __fmul_rn(exp2_ftz(fmaf(lq, kLog2e, nmlq)), invq);
        return fmaxf(__fsub_rn(p, q), 0.f);
    }
    // The same weights for two neighbouring entries, two per instruction
    // (each lane rounds exactly as the scalar form does).
    __device__ float2 pair(float2 lp, float2 lq) const {
        const float2 l2 = make_float2(kLog2e, kLog2e);
        const float2 xp = __ffma2_rn(lp, l2, make_float2(nmlp, nmlp));
        const float2 p = __fmul2_rn(make_float2(exp2_ftz(xp.x), exp2_ftz(xp.y)), make_float2(invp, invp));
        if (!resid) return p;
        const float2 xq = __ffma2_rn(lq, l2, make_float2(nmlq, nmlq));
        const float2 q = __fmul2_rn(make_float2(exp2_ftz(xq.x), exp2_ftz(xq.y)), make_float2(invq, invq));
        const float2 d = __ffma2_rn(q, make_float2(-1.f, -1.f), p);  // p - q, one rounding
        return make_float2(fmaxf(d.x, 0.f), fmaxf(d.y, 0.f));
    }
};

constexpr int kCkpt = 4;  // checkpoints of a thread's running sum over its run (the draw)

// Walk the run [e_lo, e_hi) of a row in index order, accumulating the weights
// in one sequential fp32 chain that starts at part0, and return the chain's
// value. `last` gets the last entry with a positive weight. With FIND, `first`
// gets the first entry whose position base + chain (rounded as
// fl(P + fl(T + chain))) exceeds thr with a positive weight, and the walk
// stops there. ck (not FIND): the chain's value before load unit i of the run
// is stored at ck[(i / seg) kAT] for i a multiple of seg (shared memory).
template <typename T, bool VEC, bool FIND>
__device__ float run_weights(const T *prow, const T *qrow, int e_lo, int e_hi, const Weigher &wf, float P, float Tk,
                             float thr, int &first, int &last, float part0 = 0.f, float *ck = nullptr, int seg = 1) {
    float part = part0;
    auto visit = [&](float w, int e) {
        part = __fadd_rn(part, w);
        if (w > 0.f) {
            last = e;
            if (FIND && first < 0 && __fadd_rn(P, __fadd_rn(Tk, part)) > thr) first = e;
        }
    };
    if (VEC) {
        // FIND: groups of two vectors per row, the next group's loads issued
        // before the current group is consumed
        constexpr int W = Logit<T>::W, G = 2;
        const uint4 *pv = reinterpret_cast<const uint4 *>(prow);
        const uint4 *qv = reinterpret_cast<const uint4 *>(qrow);
        const int vlo = e_lo / W, vhi = e_hi / W;
        uint4 cp[G], cq[G], np_[G], nq[G];
        auto fetch = [&](uint4 (&rp)[G], uint4 (&rq)[G], int v) {
#pragma unroll
            for (int k = 0; k < G; ++k) {
                const bool ok = v + k < vhi;
                rp[k] = ok ? __ldg(pv + v + k) : make_uint4(0, 0, 0, 0);
                rq[k] = ok && wf.resid ? __ldg(qv + v + k) : make_uint4(0, 0, 0, 0);
            }
        };
        if constexpr (!FIND) {
            // the sum pass: four vectors of each row per round, all in flight together (the
            // same registers as two rounds ahead of two)
            constexpr int G4 = 4;
            for (int v = vlo; v < vhi; v += G4) {
                uint4 rp[G4], rq[G4];
#pragma unroll
                for (int k = 0; k < G4; ++k) {
                    const bool ok = v + k < vhi;
                    rp[k] = ok ? __ldg(pv + v + k) : make_uint4(0, 0, 0, 0);
                    rq[k] = ok && wf.resid ? __ldg(qv + v + k) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int k = 0; k < G4; ++k) {
                    if (v + k >= vhi) break;
                    if (ck != nullptr && (v + k - vlo) % seg == 0) ck[(v + k - vlo) / seg * kAT] = part;
#pragma unroll
                    for (int q = 0; q < W / 2; ++q) {
                        const float2 w = wf.pair(Logit<T>::pair(rp[k], q), Logit<T>::pair(rq[k], q));
                        const int e = (v + k) * W + 2 * q;
                        visit(w.x, e);
                        visit(w.y, e + 1);
                    }
                }
            }
            return part;
        }
        if (vlo < vhi) fetch(cp, cq, vlo);
        for (int v = vlo; v < vhi; v += G) {
            if (FIND && first >= 0) break;
            if (v + G < vhi) fetch(np_, nq, v + G);
#pragma unroll
            for (int k = 0; k < G; ++k) {
                if (v + k >= vhi) break;
#pragma unroll
                for (int q = 0; q < W / 2; ++q) {
                    const float2 w = wf.pair(Logit<T>::pair(cp[k], q), Logit<T>::pair(cq[k], q));
                    const int e = (v + k) * W + 2 * q;
                    visit(w.x, e);
                    visit(w.y, e + 1);
                }
            }
#pragma unroll
            for (int k = 0; k < G; ++k) {
                cp[k] = np_[k];
                cq[k] = nq[k];
            }
        }
    } else {
        for (int e = e_lo; e < e_hi; ++e) {
            if (FIND && first >= 0) break;
            if (!FIND && ck != nullptr && (e - e_lo) % seg == 0) ck[(e - e_lo) / seg * kAT] = part;
            visit(wf(Logit<T>::one(prow + e), wf.resid ? Logit<T>::one(qrow + e) : 0.f), e);
        }
    }
    return part;
}

template <typename T, bool SAMPLE, bool VEC>
__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kAT, 4) ssm_accept_kernel(const AArgs a) {
    __shared__ float2 wpart[2 * kGroup][kAWarps];  // this step's rows: one partial per warp
    __shared__ float2 cpart[2][2 * kGroup];        // [step parity][row]: this CTA's partials, read by the cluster
    __shared__ float2 fin[2 * kGroup];             // this step's row statistics for the sequence
    __shared__ float wsum[kAWarps];
    __shared__ float cW;                  // this CTA's total weight (read by the whole cluster)
    __shared__ int s_rej, s_bad, s_owner, s_first, s_last;
    __shared__ float s_P, s_thr;
    __shared__ float ckpt[kCkpt * kAT];  // the draw: each thread's running sum at checkpoints of its run

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = (int)(blockIdx.x / kCl);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K, V = a.V;
    const T *tl = static_cast<const T *>(a.tl) + (int64_t)b * (K + 1) * V;
    const T *ql = SAMPLE ? static_cast<const T *>(a.ql) + (int64_t)b * K * V : nullptr;
    const int lo = min(rank * a.slice, V), hi = min(lo + a.slice, V);
    constexpr int W = VEC ? Logit<T>::W : 1;

    // ---- the logits at the draft tokens and the uniforms, which the
    // acceptance rule reads: loaded first (warp 0, lane t for token t) so that
    // their latency hides behind the first row pass.
    int pre_x = -1;
    float pre_lp = 0.f, pre_lq = 0.f, pre_u = 0.f;
    if (warp == 0 && lane < K) {
        pre_x = a.drafts[(int64_t)b * K + lane];
        if (SAMPLE) pre_u = a.u[(int64_t)b * (K + 1) + lane];
        if (SAMPLE && pre_x >= 0 && pre_x < V) {
            pre_lp = Logit<T>::one(tl + (int64_t)lane * V + pre_x);
            pre_lq = Logit<T>::one(ql + (int64_t)lane * V + pre_x);
        }
    }

    // ---- steps t = 0, 1, ...: the statistics of verifier row t (and draft
    // row t), then the decision on draft token t. The first rejection ends
    // the walk: rows past it are never read. Every CTA combines the cluster's
    // partials in rank order, so all take the same decisions.
    using Bt = Batch<T, VEC>;
    using Acc = typename std::conditional<SAMPLE, SoftAcc, ArgAcc>::type;
    const int ulo = lo / W, uhi = hi / W;  // slice in load units (vectors, or elements)
    // Step: tokens t0 .. t0 + ng - 1; row 2i is verifier row t0 + i, row
    // 2i + 1 draft row t0 + i (sampling, t0 + i < K).
    int j = K, badj = 0, jrow = 0;
    for (int t0 = 0; t0 <= K; t0 += kGroup) {
        const int ng = min(kGroup, K + 1 - t0);
        for (int i = 0; i < ng; ++i) {
            const int nr = (SAMPLE && t0 + i < K) ? 2 : 1;
            for (int r = 0; r < nr; ++r) {
                const T *src = (r == 0 ? tl : ql) + (int64_t)(t0 + i) * V;
                Acc acc;
                for (int u0 = ulo + tid; u0 < uhi; u0 += Bt::S * kAT) {
                    Bt bt;
                    bt.load(src, u0, uhi);
                    acc.push(bt);
                }
                const float2 out = acc.warp_total();
                if (lane == 0) wpart[2 * i + r][warp] = out;
            }
        }
        __syncthreads();
        const int par = (t0 / kGroup) & 1;
        auto rowvalid = [&](int q) { return q / 2 < ng && (q % 2 == 0 || (SAMPLE && t0 + q / 2 < K)); };
        if (tid < 2 * kGroup && rowvalid(tid)) {
            float2 c = wpart[tid][0];
            for (int w = 1; w < kAWarps; ++w) {
                const float2 o = wpart[tid][w];
                if (SAMPLE) {
                    soft_combine(c.x, c.y, o.x, o.y);
                } else {
                    int i = __float_as_int(c.y);
                    arg_combine(c.x, i, o.x, __float_as_int(o.y));
                    c.y = __int_as_float(i);
                }
            }
            cpart[par][tid] = c;
        }
        cluster.sync();  // every CTA's partials of this step are published
        if (tid < 2 * kGroup && rowvalid(tid)) {
            float2 c = *cluster.map_shared_rank(&cpart[par][tid], 0);
            for (int r = 1; r < kCl; ++r) {
                const float2 o = *cluster.map_shared_rank(&cpart[par][tid], r);
                if (SAMPLE) {
                    soft_combine(c.x, c.y, o.x, o.y);
                } else {
                    int i = __float_as_int(c.y);
                    arg_combine(c.x, i, o.x, __float_as_int(o.y));
                    c.y = __int_as_float(i);
                }
            }
            fin[tid] = c;
        }
        __syncthreads();
        if (warp == 0) {  // lane t holds token t's prefetched values
            bool rej = false, bad = false;
            const int i = lane - t0;
            if (i >= 0 && i < ng && lane < K) {
                bad = pre_x < 0 || pre_x >= V;
                if (bad) {
                    rej = true;
                } else if (!SAMPLE) {
                    rej = __float_as_int(fin[2 * i].y) != pre_x;
                } else {
                    const float2 fp = fin[2 * i], fq = fin[2 * i + 1];
                    const float ep = exp2_ftz(fmaf(pre_lp, kLog2e, -(fp.x * kLog2e)));
                    const float eq = exp2_ftz(fmaf(pre_lq, kLog2e, -(fq.x * kLog2e)));
                    const float p = __fdiv_rn(ep, fp.y), q = __fdiv_rn(eq, fq.y);
                    const float ratio = q > 0.f ? __fdiv_rn(p, q) : INFINITY;
                    rej = !(pre_u < ratio);
                }
            }
            const unsigned m = __ballot_sync(~0u, rej);
            if (lane == 0) {
                s_rej = m != 0u ? __ffs(m) - 1 : -1;  // the first rejected token of the step, if any
            }
            const int first = m != 0u ? __ffs(m) - 1 : 0;
            const int fb = __shfl_sync(~0u, bad ? 1 : 0, first);
            if (lane == 0) s_bad = fb;
        }
        __syncthreads();
        if (s_rej >= 0) {  // the same in every CTA of the cluster
            j = s_rej;
            badj = s_bad;
            jrow = 2 * (j - t0);
            break;
        }
        if (t0 + ng > K) {  // every draft token accepted: row K gives the bonus token
            jrow = 2 * (K - t0);
            break;
        }
    }
    if (tid == 0 && rank == 0) {
        a.accept_len[b] = j;
        if (badj && a.dev_status != nullptr) atomicOr(a.dev_status, SSM_STATUS_BAD_TOKEN);
        if (!SAMPLE) a.next_token[b] = __float_as_int(fin[jrow].y);
    }
    if (!SAMPLE) {
        cluster.sync();  // no CTA leaves while another may still read its partials
        return;
    }

    // ---- the draw (sampling): the next token, by inverse CDF at u_K over row j
    Weigher wf;
    wf.resid = j < K && !badj;
    {
        const float2 fp = fin[jrow];
        wf.nmlp = -(fp.x * kLog2e);
        wf.invp = __frcp_rn(fp.y);
        const float2 fq = wf.resid ? fin[jrow + 1] : make_float2(0.f, 1.f);
        wf.nmlq = -(fq.x * kLog2e);
        wf.invq = __frcp_rn(fq.y);
    }
    const T *prow = tl + (int64_t)j * V;
    const T *qrow = wf.resid ? ql + (int64_t)j * V : prow;
    const int n = hi - lo;
    const int per = ((n + kAT - 1) / kAT + W - 1) / W * W;  // a thread's contiguous run
    const int e_lo = min(lo + tid * per, hi), e_hi = min(e_lo + per, hi);
    int dummy0 = -1, lastpos = -1;
    // the run in load units (vectors, or elements), cut into at most kCkpt segments
    const int units = VEC ? (e_hi - e_lo) / W : e_hi - e_lo;
    const int seg = units > 0 ? (units + kCkpt - 1) / kCkpt : 1;
    const float s_k = run_weights<T, VEC, false>(prow, qrow, e_lo, e_hi, wf, 0.f, 0.f, 0.f, dummy0, lastpos, 0.f,
                                                 ckpt + tid, seg);
    // exclusive prefix of the runs over the CTA
    float incl = s_k;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(~0u, incl, off);
        if (lane >= off) incl = __fadd_rn(incl, o);
    }
    float excl = __shfl_up_sync(~0u, incl, 1);
    if (lane == 0) excl = 0.f;
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    float before = 0.f;
    for (int w = 0; w < warp; ++w) before = __fadd_rn(before, wsum[w]);
    const float Tk = __fadd_rn(before, excl);
    if (tid == 0) {
        float tot = 0.f;
        for (int w = 0; w < kAWarps; ++w) tot = __fadd_rn(tot, wsum[w]);
        cW = tot;
        s_first = kNoIndex;
        s_last = -1;
    }
    cluster.sync();
    if (tid == 0) {
        // the cluster prefix, in rank order: the same chain in every CTA
        float P = 0.f, Pmine = 0.f;
        float Wr[kCl], Q[kCl];
        for (int r = 0; r < kCl; ++r) {
            Wr[r] = *cluster.map_shared_rank(&cW, r);
            if (r == rank) Pmine = P;
            P = __fadd_rn(P, Wr[r]);
            Q[r] = P;
        }
        const float thr = __fmul_rn(a.u[(int64_t)b * (K + 1) + K], P);
        int owner = -1;
        for (int r = 0; r < kCl && owner < 0; ++r)
            if (Q[r] > thr) owner = r;
        if (owner < 0)
            for (int r = kCl - 1; r >= 0 && owner < 0; --r)
                if (Wr[r] > 0.f) owner = r;
        s_owner = owner;
        s_P = Pmine;
        s_thr = thr;
        if (owner < 0 && rank == 0) a.next_token[b] = V - 1;  // no positive weight anywhere
    }
    cluster_arrive();  // this CTA's remote reads are done
    __syncthreads();
    if (s_owner == rank) {
        const float P = s_P, thr = s_thr;
        const float hiK = __fadd_rn(P, __fadd_rn(Tk, s_k));
        if (s_k > 0.f) {
            if (hiK > thr) atomicMin(&s_first, tid);
            atomicMax(&s_last, tid);
        }
        __syncthreads();
        const int who = s_first != kNoIndex ? s_first : s_last;
        if (tid == who) {
            // The test is monotone in the running sum, so no entry before the first segment whose end
            // passes it can pass: the walk starts there, from the chain's exact value at that point.
            const int nseg = (units + seg - 1) / seg;
            int sg = 0;
            while (sg < nseg) {
                const float end = sg + 1 < nseg ? ckpt[(sg + 1) * kAT + tid] : s_k;
                if (__fadd_rn(P, __fadd_rn(Tk, end)) > thr) break;
                ++sg;
            }
            int first = -1, last = -1;
            if (sg < nseg)
                run_weights<T, VEC, true>(prow, qrow, e_lo + sg * seg * (VEC ? W : 1), e_hi, wf, P, Tk, thr, first,
                                          last, ckpt[sg * kAT + tid]);
            a.next_token[b] = first >= 0 ? first : lastpos;
        }
    }
    cluster_wait();  // no CTA leaves while another may still read its total
}

// ----------------------------------------------------------------------------- host side

bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Span {
    uintptr_t lo, hi;
};

Span span_of(const void *p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Span{lo, lo + static_cast<uintptr_t>(bytes)};
}

bool overlap(const Span &x, const Span &y) { return x.lo < y.hi && y.lo < x.hi; }

template <typename T, bool SAMPLE, bool VEC>
cudaError_t launch_accept(const AArgs &a, int batch, cudaStream_t s) {
    ssm_accept_kernel<T, SAMPLE, VEC><<<(unsigned)batch * kCl, kAT, 0, s>>>(a);
    return cudaGetLastError();
}

template <bool SAMPLE>
cudaError_t launch_dtype(int dtype, bool vec, const AArgs &a, int batch, cudaStream_t s) {
    if (dtype == SSM_BF16)
        return vec ? launch_accept<__nv_bfloat16, SAMPLE, true>(a, batch, s)
                   : launch_accept<__nv_bfloat16, SAMPLE, false>(a, batch, s);
    return vec ? launch_accept<float, SAMPLE, true>(a, batch, s) : launch_accept<float, SAMPLE, false>(a, batch, s);
}

int run_accept(const ssm_accept_desc_t *d, bool sample, const void *tl, const void *ql, const int32_t *drafts,
               const float *u, int32_t *accept_len, int32_t *next_token, uint32_t *dev_status, void *stream) {
    if (d == nullptr) return SSM_ERR_NULL;
    if (d->batch < 0 || d->ntok < 1 || d->ntok > SSM_ACCEPT_MAX_NTOK || d->vocab < 1 ||
        d->vocab > SSM_ACCEPT_MAX_VOCAB)
        return SSM_ERR_SHAPE;
    if (d->logit_dtype != SSM_F32 && d->logit_dtype != SSM_BF16) return SSM_ERR_UNSUPPORTED;
    if ((int64_t)d->batch * kCl > INT_MAX) return SSM_ERR_SHAPE;
    if (d->batch == 0) return SSM_OK;
    if (tl == nullptr || drafts == nullptr || accept_len == nullptr || next_token == nullptr) return SSM_ERR_NULL;
    if (sample && (ql == nullptr || u == nullptr)) return SSM_ERR_NULL;
    const int64_t es = d->logit_dtype == SSM_BF16 ? 2 : 4;
    if (!aligned_to(tl, es) || !aligned_to(drafts, 4) || !aligned_to(accept_len, 4) || !aligned_to(next_token, 4))
        return SSM_ERR_ALIGN;
    if (sample && (!aligned_to(ql, es) || !aligned_to(u, 4))) return SSM_ERR_ALIGN;
    if (dev_status != nullptr && !aligned_to(dev_status, 4)) return SSM_ERR_ALIGN;

    const int64_t Bn = d->batch, K = d->ntok, V = d->vocab;
    Span in[4];
    int nin = 0;
    in[nin++] = span_of(tl, Bn * (K + 1) * V * es);
    in[nin++] = span_of(drafts, Bn * K * 4);
    if (sample) {
        in[nin++] = span_of(ql, Bn * K * V * es);
        in[nin++] = span_of(u, Bn * (K + 1) * 4);
    }
    Span out[3];
    int nout = 0;
    out[nout++] = span_of(accept_len, Bn * 4);
    out[nout++] = span_of(next_token, Bn * 4);
    if (dev_status != nullptr) out[nout++] = span_of(dev_status, 4);
    for (int i = 0; i < nout; ++i) {
        for (int k = 0; k < nin; ++k)
            if (overlap(out[i], in[k])) return SSM_ERR_ALIAS;
        for (int k = 0; k < nout; ++k)
            if (k != i && overlap(out[i], out[k])) return SSM_ERR_ALIAS;
    }

    const int W = d->logit_dtype == SSM_BF16 ? 8 : 4;
    const bool vec = aligned_to(tl, 16) && (!sample || aligned_to(ql, 16)) && (V * es) % 16 == 0;
    const int unit = vec ? W : 1;
    AArgs a;
    a.tl = tl;
    a.ql = ql;
    a.drafts = drafts;
    a.u = u;
    a.accept_len = accept_len;
    a.next_token = next_token;
    a.dev_status = dev_status;
    a.K = d->ntok;
    a.V = d->vocab;
    const int64_t per = (V + kCl - 1) / kCl;
    a.slice = (int)((per + unit - 1) / unit * unit);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaError_t e = sample ? launch_dtype<true>(d->logit_dtype, vec, a, d->batch, s)
                                 : launch_dtype<false>(d->logit_dtype, vec, a, d->batch, s);
    if (e != cudaSuccess) {
        ssm_internal::set_last_cuda_error((int)e);
        return SSM_ERR_CUDA;
    }
    return SSM_OK;
}

}  // namespace

extern "C" {

int ssm_accept_greedy(const ssm_accept_desc_t *desc, const void *target_logits, const int32_t *draft_tokens,
                      int32_t *accept_len, int32_t *next_token, uint32_t *dev_status, void *stream) {
    return run_accept(desc, false, target_logits, nullptr, draft_tokens, nullptr, accept_len, next_token, dev_status,
                      stream);
}

int ssm_accept_sample(const ssm_accept_desc_t *desc, const void *target_logits, const void *draft_logits,
                      const int32_t *draft_tokens, const float *uniform, int32_t *accept_len, int32_t *next_token,
                      uint32_t *dev_status, void *stream) {
    return run_accept(desc, true, target_logits, draft_logits, draft_tokens, uniform, accept_len, next_token,
                      dev_status, stream);
}

}  // extern "C"
