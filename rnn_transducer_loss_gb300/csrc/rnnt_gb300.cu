// rnnt_gb300.cu -- fused RNN-T loss forward+backward for GB300 (sm_103a).
//
// Device pipeline of one rnnt_loss_fused call (all on the caller's stream):
//   k_prepare   1 CTA: validates lengths/targets, exclusive int64 scan of
//               T_b*(U_b+1) (row offsets), largest-lattice-first sample order.
//               Replaces the host-side largest-task-first balancer of the
//               rnnt-loss-ascend README (架构设计 "Host 侧").
//   k_row_*     one pass over the logits: per row the log-softmax denominator
//               (max, then sum of exponentials, group-shuffle reductions) and
//               the blank / target transition probabilities, stored per
//               lattice node in anti-diagonal-packed order so that each
//               step of the DP's anti-diagonal sweep (README 对角线遍历 α/β)
//               reads and writes one contiguous run.  With the in-kernel log-softmax off only the two needed
//               elements of a row are read.
//   k_dp        one CTA per (sample, direction): the forward (alpha)
//               recursion over anti-diagonals d = 0..T+U-1, or the backward
//               (beta) one from the end, on up to 4 warps; lattice columns
//               per lane, the neighbouring column's value by warp shuffle.
//   k_grad      per row the occupancy and the blank/label arc posteriors from
//               alpha, beta and P(y|x) (README 核心梯度融合公式), then one
//               read + one write of the logits: grad_k = p_k*occ -
//               [k=blank]*post_blank - [k=y]*post_label, clip, reduction
//               scale, store in the input dtype (may alias the logits).
//               Rows whose occupancy is too small to change any output value
//               are written as zeros without reading the logits.  Its last
//               CTA runs the alpha/beta loss cross-check (README 精度保证
//               "双 loss 互校验"), the deterministic reduction and the status
//               word (k_finalize does so for a loss-only call).
// One persistent cooperative kernel (k_main) runs all of this as tasks when
// the shape allows; the kernels above are the per-stage schedule.
//
// Numerics.  The DP runs in the probability domain on extended-range
// numbers m * 2^e (m in [1,2) as float, e as int32): a product is one
// float multiply and an integer add, a sum aligns the exponents exactly and
// does one fused multiply-add.  Every step therefore rounds only with
// round-to-nearest multiplies/adds and nothing underflows, which is the
// same protection the README's log-domain recursion ("全程在 log 域") is
// after, without evaluating a transcendental function per lattice node.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#include <cooperative_groups.h>

#include <algorithm>
#include <mutex>
#include <type_traits>

#include "rnnt_gb300.h"

namespace {

constexpr float kLog2e = 1.4426950216293335f;     // float(log2 e)
constexpr float kLog2eLo = 1.925962989e-8f;        // log2 e - kLog2e
constexpr float kLn2 = 0.6931471824645996f;
constexpr float kSqrt2 = 1.4142135381698608f;
constexpr double kLn2d = 0.69314718055994530942;
constexpr int kMaxW = RNNT_MAX_TARGET_LENGTH + 1;
constexpr int kZeroExp = -(1 << 29);               // exponent of an extended-range zero
// Transition records store exponents + kEdgeBias, so an all-zero record is a
// zero probability (m = 0, e = kZeroExp); the DP's zero-filled loads rely on it.
constexpr int kEdgeBias = 1 << 29;

enum : int {
    ERR_LENGTH = 1,
    ERR_ROWS = 2,
    ERR_TARGET = 4,
    ERR_MISMATCH = 8,
    ERR_NONFINITE = 16,
    ERR_TIMEOUT = 32,
    ERR_INTERNAL = 64,   // a configuration the launching host code rules out

};

// ---------------------------------------------------------------- workspace
constexpr int kTaskRows = 256;   // rows per row / gradient task of the persistent kernel

struct Layout {
    size_t err, off, order, lossa, lossb, pm, pe, lse2, edge, alpha, beta;
    size_t rtasks, rdone, dpdone, dpclaim, tasks, total;
    int64_t max_tasks;
};

// Upper bound of the persistent kernel's task count: per sample its row
// chunks, one DP task and its gradient chunks.
__host__ __device__ inline int64_t max_tasks_for(int B, int64_t rows) {
    return 2 * (rows / kTaskRows + B) + B;
}

__host__ __device__ inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline Layout ws_layout(int B, int64_t rows) {
    Layout L;
    size_t p = 0;
    const size_t R = (size_t)rows;
    L.err = p;   p = al256(p + 256);
    L.off = p;   p = al256(p + sizeof(int64_t) * (size_t)(B + 1));
    L.order = p; p = al256(p + sizeof(int32_t) * (size_t)B);
    L.lossa = p; p = al256(p + sizeof(double) * (size_t)B);
    L.lossb = p; p = al256(p + sizeof(double) * (size_t)B);
    L.pm = p;    p = al256(p + sizeof(float) * (size_t)B);
    L.pe = p;    p = al256(p + sizeof(int32_t) * (size_t)B);
    L.lse2 = p;  p = al256(p + sizeof(float) * R);
    L.edge = p;  p = al256(p + sizeof(int4) * R);
    L.alpha = p; p = al256(p + sizeof(int2) * R);
    L.beta = p;  p = al256(p + sizeof(int2) * R);
    L.max_tasks = max_tasks_for(B, rows);
    L.rtasks = p; p = al256(p + sizeof(int32_t) * (size_t)B);
    L.rdone = p;  p = al256(p + sizeof(int32_t) * (size_t)B);
    L.dpdone = p; p = al256(p + sizeof(int32_t) * (size_t)B);
    L.dpclaim = p; p = al256(p + sizeof(int32_t) * (size_t)B);
    L.tasks = p;  p = al256(p + 2 * sizeof(int4) * (size_t)L.max_tasks);
    L.total = p;
    return L;
}

// Rows of at least this many bytes take a separate record pass before the
// per-stage gradient kernel (measured on 20 KB rows: forming each row's record
// inside the gradient kernel stalls its warp on a chain of dependent loads).
constexpr size_t kLongRowBytes = 8192;
__host__ __device__ inline bool long_rows(int V, int dt) {
    return (size_t)V * (dt == RNNT_F32 ? 4 : 2) >= kLongRowBytes;
}
// Workspace: the common layout, plus for long rows one gradient record
// (float4) per row after it.
__host__ __device__ inline size_t ws_total(int B, int64_t rows, int V, int dt) {
    return ws_layout(B, rows).total + (long_rows(V, dt) ? al256(sizeof(float4) * (size_t)rows) : 0);
}

// Workspace of the multi-blank kernels: the common layout plus one
// extended-range probability per big blank and lattice node.
__host__ __device__ inline size_t ws_total_mb(int B, int64_t rows, int K) {
    return ws_layout(B, rows).total + al256(sizeof(int2) * (size_t)K * (size_t)rows);
}

struct Params {
    const void* logits;
    void* grad;
    int64_t rows;
    int V;
    int dt;
    const int32_t* targets;
    int S;
    const int32_t* Tl;
    const int32_t* Ul;
    int B;
    int blank;
    float clamp;      // +inf when clipping is off
    float scale;      // reduction scale applied to the gradient
    float skip2;      // log2-occupancy below which a gradient row is exactly zero
    float lscale;     // log2(scale)
    int fused;
    int red;
    float fe;         // FastEmit weight: label-emission gradient terms scaled by 1 + fe
    float fe_l2;      // log2(1 + fe)
    int padded;       // logits/grad are the padded (B, maxT, maxW, V) tensor
    int maxT, maxW;   // padded layout: frames and lattice columns of a sample slot
    // Multi-blank transducer: K big blanks (output bb_id[i], bb_dur[i] frames),
    // every transition probability times bb_c = e^-sigma; pbb[i * rows + node]
    // holds big blank i's probability at a node (extended range, biased exponent).
    int K;
    int bb_id[RNNT_MAX_BIG_BLANKS];
    int bb_dur[RNNT_MAX_BIG_BLANKS];
    float bb_c;
    int2* pbb;
    int stage_bytes;  // per-stage shared-memory row buffer of the TMA-staged passes
    int zero_off;     // persistent kernel: shared-memory offset of a zeroed buffer ...
    int zero_rows;    // ... of zero_rows gradient rows, the source of zero-row bulk stores
    // Calls without the in-kernel log-softmax: extra CTAs of the recursion
    // launch zero the whole gradient buffer (zfill bytes; zcta CTAs at most,
    // each with a zeroed shared buffer of zbuf bytes), and the gradient pass
    // then writes only the blank and label elements.  zfill = 0: off.
    int64_t zfill;
    int zcta, zbuf;
    float* loss;
    float* loss_red;
    int32_t* status;
    // workspace views
    int32_t* err;
    int64_t* off;
    int32_t* order;
    double* lossa;
    double* lossb;
    float* pm;        // P(y|x) of each sample, extended range
    int32_t* pe;
    float* lse2;      // per row (row order): log2 sum_k 2^(h_k log2 e)
    float4* info;     // long rows only: per row the gradient record (k_combine)
    int4* edge;       // per node (node_index order): {p_blank.m, p_blank.e, p_label.m, p_label.e}
    int2* alpha;      // per node (node_index order): {m, e}
    int2* beta;
    // persistent-kernel scheduler (err[1] = next task, err[2] = task count)
    int32_t* rtasks;  // row tasks per sample
    int32_t* rdone;   // finished row tasks per sample
    int32_t* dpdone;  // DP finished flag per sample
    int32_t* dpclaim; // DP started (claimed) flag per sample
    int n_dp_sms;     // SMs whose CTAs only run DP tasks
    int build_tasks;  // the preparation builds the persistent kernel's task list
    int4* tasks;      // 2 per task: {kind | sample << 2, first row in sample, rows, T},
                      // {U, 0, first row of the sample (int64, low, high)}
    int4* trace;      // optional per-task trace records (see rnnt_set_trace), or null
    int64_t trace_cap;
};

// ---------------------------------------------------------------- helpers
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Number of lattice nodes (t,u), 0<=t<T, 0<=u<W, with t+u < d: first index
// of anti-diagonal d in the per-node arrays (inclusion-exclusion over the
// rectangle).
__device__ __forceinline__ int64_t tri(int64_t n) { return n > 0 ? n * (n + 1) / 2 : 0; }
__device__ __forceinline__ int64_t diag_start(int d, int T, int W) {
    return tri(d) - tri((int64_t)d - T) - tri((int64_t)d - W) + tri((int64_t)d - T - W);
}
// Index of node (t,u) relative to its sample's first record in the per-node
// arrays (transition records, alpha, beta): anti-diagonal-packed, so each
// diagonal d = t+u is one contiguous run ordered by t.
// When T + W <= 65536 every triangular number involved is below 2^32 and the
// index below 2^31, so 32-bit unsigned arithmetic gives it exactly.
__device__ __forceinline__ unsigned tri32(int n) {
    return n > 0 ? ((unsigned)n * (unsigned)(n + 1)) >> 1 : 0u;
}
__device__ __forceinline__ int64_t node_index(int t, int u, int T, int U) {
    const int d = t + u;
    if (T + U < 65536) {
        const int W = U + 1;
        const unsigned ds = tri32(d) - tri32(d - T) - tri32(d - W) + tri32(d - T - W);
        return (int64_t)(int)(ds + (unsigned)(t - max(0, d - U)));
    }
    return diag_start(d, T, U + 1) + (t - max(0, d - U));
}

__device__ __forceinline__ int find_sample(const int64_t* off, int B, int64_t r) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldcg(off + mid) <= r) lo = mid; else hi = mid;
    }
    return lo;
}

// The same by a whole warp (every lane calls it, same r): a 32-way search, one
// round of loads per factor of 32 in B, all lanes return the sample.
__device__ __forceinline__ int find_sample_warp(const int64_t* off, int B, int64_t r) {
    const int lane = threadIdx.x & 31;
    int lo = 0, n = B;   // off[lo] <= r < off[lo + n]
    while (n > 1) {
        const int step = (n + 31) / 32;
        const int idx = lo + lane * step;
        const bool le = idx < lo + n && __ldcg(off + idx) <= r;
        const unsigned bal = __ballot_sync(0xffffffffu, le);
        const int k = 31 - __clz(bal);
        lo += k * step;
        n = min(step, n - k * step);
    }
    return lo;
}

// Logits / gradient row holding lattice row r (compact numbering) of sample b,
// whose compact rows start at o and whose lattice is W nodes wide: r itself in
// the compact layout, (b*maxT + t)*maxW + u in the padded one.
__device__ __forceinline__ int64_t lrow_s(const Params& p, int64_t r, int b, int64_t o, int W) {
    if (!p.padded) return r;
    const unsigned i = (unsigned)(r - o);
    const int t = (int)(i / (unsigned)W), u = (int)(i - (unsigned)t * W);
    return ((int64_t)b * p.maxT + t) * p.maxW + u;
}
// Lattice nodes of the batch (compact rows): the logits' row count in the
// compact layout, sum_b T_b*(U_b+1) (written earlier in this call) in the
// padded one.
__device__ __forceinline__ int64_t nodes(const Params& p) {
    return p.padded ? __ldcg(p.off + p.B) : p.rows;
}
// The same with the sample looked up (offsets written earlier in this call).
__device__ __forceinline__ int64_t lrow(const Params& p, int64_t r) {
    if (!p.padded) return r;
    const int b = find_sample(p.off, p.B, r);
    return lrow_s(p, r, b, __ldcg(p.off + b), __ldg(p.Ul + b) + 1);
}
// Rows are visited in increasing order; step to r's sample, searching only on a change.
__device__ __forceinline__ int advance_sample(const int64_t* off, int B, int b, int64_t r) {
    return (__ldcg(off + b + 1) <= r) ? find_sample(off, B, r) : b;
}

// ------------------------------------------------ extended-range arithmetic
// 2^f for f in [0,1) as sqrt(2) * exp(g), g = (f - 1/2) ln 2, |g| <= 0.347,
// with the Taylor series of exp truncated after g^9 (remainder < 3e-10).
__device__ __forceinline__ float exp_taylor(float g) {
    float q = 1.0f / 362880.0f;
    q = fmaf(q, g, 1.0f / 40320.0f);
    q = fmaf(q, g, 1.0f / 5040.0f);
    q = fmaf(q, g, 1.0f / 720.0f);
    q = fmaf(q, g, 1.0f / 120.0f);
    q = fmaf(q, g, 1.0f / 24.0f);
    q = fmaf(q, g, 1.0f / 6.0f);
    q = fmaf(q, g, 0.5f);
    q = fmaf(q, g, 1.0f);
    return fmaf(q, g, 1.0f);
}

// Renormalise m * 2^e to m in [1,2) (m > 0 finite), or leave a zero alone.
__device__ __forceinline__ void xf_norm(float& m, int& e) {
    const int bits = __float_as_int(m);
    const int ex = (m != 0.0f) ? (bits >> 23) - 127 : 0;
    m = __int_as_float(bits - (ex << 23));
    e += ex;
}

// 2^(xh + xl) as m * 2^e, m in [1,2); xl is a small correction (|xl| < 1e-3).
__device__ __forceinline__ void xf_exp2(float xh, float xl, float& m, int& e) {
    if (!(xh > -1.0e8f)) {   // -inf (a zero probability) and anything below 2^-1e8
        m = 0.0f;
        e = kZeroExp;
        return;
    }
    const float n = floorf(fminf(xh, 1.0e8f));
    const float f = xh - n;                      // exact, in [0, 1)
    m = exp_taylor(fmaf(f - 0.5f, kLn2, xl * kLn2)) * kSqrt2;
    e = (int)n;
    xf_norm(m, e);
}

// p = 2^((h - M) log2 e) / s with the exponent carried in two floats.
__device__ __forceinline__ void xf_prob(float h, float M, float s, float& m, int& e) {
    const float d = h - M;                       // TwoSum(h, -M)
    const float bb = d - h;
    const float derr = (h - (d - bb)) + (-M - bb);
    const float xh = d * kLog2e;
    const float xl = fmaf(d, kLog2e, -xh) + fmaf(derr, kLog2e, d * kLog2eLo);
    xf_exp2(xh, xl, m, e);
    if (m != 0.0f) {
        m = m / s;
        xf_norm(m, e);
    }
}

// Product of two extended-range numbers.  Exponents stay >= kZeroExp because
// every sum below clamps its result, so a product of two zeros (2*kZeroExp)
// cannot overflow.
__device__ __forceinline__ void xf_mul(float am, int ae, float pm, int pe, float& m, int& e) {
    m = am * pm;
    e = ae + pe;
}

// (m1 2^e1) + (m2 2^e2): exact alignment by the exponent difference, one FMA.
// With NORM the mantissa is brought back to [1,2); without it the mantissa may
// grow (by at most 2^3 per step: inputs are products of two mantissas below
// 2^w and 2 each), which the exponent alignment tolerates exactly.
template <bool NORM = true>
__device__ __forceinline__ void xf_add(float m1, int e1, float m2, int e2, float& m, int& e) {
    const bool first = e1 >= e2;
    const float big = first ? m1 : m2, small = first ? m2 : m1;
    const int E = first ? e1 : e2;
    const int k = first ? e2 - e1 : e1 - e2;                   // <= 0
    const float sc = __int_as_float(max(k + 127, 0) << 23);    // 2^k (0 below 2^-126)
    m = fmaf(small, sc, big);
    e = max(E, kZeroExp);
    if (NORM) xf_norm(m, e);
}

template <typename Tin> struct Elt;
template <> struct Elt<float> {
    static constexpr int kPerVec = 4;
    __device__ static float get(const float* p, int64_t i) { return __ldg(p + i); }
    __device__ static void unpack(const uint4& q, float* x) {
        x[0] = __uint_as_float(q.x); x[1] = __uint_as_float(q.y);
        x[2] = __uint_as_float(q.z); x[3] = __uint_as_float(q.w);
    }
    __device__ static uint4 pack(const float* g) {
        return make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                          __float_as_uint(g[3]));
    }
    __device__ static float to_f(float v) { return v; }
    __device__ static float from_f(float v) { return v; }
    __device__ static float vmax(const uint4& q) {
        return fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                     fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
    }
};
template <> struct Elt<__half> {
    static constexpr int kPerVec = 8;
    __device__ static float get(const __half* p, int64_t i) { return __half2float(__ldg(p + i)); }
    __device__ static void unpack(const uint4& q, float* x) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __half2 h = *reinterpret_cast<const __half2*>(&w[k]);
            float2 f = __half22float2(h);
            x[2 * k] = f.x;
            x[2 * k + 1] = f.y;
        }
    }
    __device__ static uint4 pack(const float* g) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __half2 h = __floats2half2_rn(g[2 * k], g[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ static float to_f(__half v) { return __half2float(v); }
    __device__ static __half from_f(float v) { return __float2half_rn(v); }
    // Exact max of 8 halves (packed compares), widened once.
    __device__ static float vmax(const uint4& q) {
        const __half2 a = __hmax2(*reinterpret_cast<const __half2*>(&q.x),
                                  *reinterpret_cast<const __half2*>(&q.y));
        const __half2 b = __hmax2(*reinterpret_cast<const __half2*>(&q.z),
                                  *reinterpret_cast<const __half2*>(&q.w));
        const float2 f = __half22float2(__hmax2(a, b));
        return fmaxf(f.x, f.y);
    }
};
// bfloat16 storage: widening to float is exact (the bits shifted up by 16).
template <> struct Elt<__nv_bfloat16> {
    static constexpr int kPerVec = 8;
    __device__ static float get(const __nv_bfloat16* p, int64_t i) {
        return __bfloat162float(__ldg(p + i));
    }
    __device__ static void unpack(const uint4& q, float* x) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
    __device__ static uint4 pack(const float* g) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(g[2 * k], g[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
    __device__ static float vmax(const uint4& q) {
        float x[8];
        unpack(q, x);
        return fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                     fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
    }
};

template <int G>
__device__ __forceinline__ unsigned group_mask() {
    if constexpr (G == 32) {
        return 0xffffffffu;
    } else {
        const unsigned lane = threadIdx.x & 31;
        return ((1u << G) - 1u) << (lane & ~(unsigned)(G - 1));
    }
}

template <int G>
__device__ __forceinline__ float group_max(float v, unsigned gm) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(gm, v, o, G));
    return v;
}
template <int G>
__device__ __forceinline__ float group_sum(float v, unsigned gm) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(gm, v, o, G);
    return v;
}

// ------------------------------------------------ TMA bulk copies + mbarriers
// Each warp of the streaming passes owns kStages shared-memory row buffers,
// each with an mbarrier; lane 0 issues one 1-D bulk copy (cp.async.bulk) per
// row, the warp waits on the barrier's phase parity.  Every wait is bounded.
#ifndef RNNT_KSTAGES
#define RNNT_KSTAGES 4
#endif
constexpr int kStages = RNNT_KSTAGES;
// Ring depth of the persistent kernel's warps: rows of 8 vectors per lane
// (4 KB) get 3 stages so that two CTAs still share an SM.
__host__ __device__ constexpr int main_stages(int NV) { return NV >= 8 ? 3 : kStages; }
constexpr int kWaitSpins = 1 << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
    return (uint32_t)__cvta_generic_to_shared(ptr);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tma_row_load(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Bulk (TMA) store of `bytes` from shared to global memory, in this thread's
// bulk group; both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void tma_store(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void tma_store_commit() {
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred q;\n mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n"
        " selp.b32 %0, 1, 0, q;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// A bounded wait gave up: set the timeout bit and, for diagnosis, record the
// first site (err[9]: 1 TMA ring, 2 DP worker waiting for rows, 3 gradient
// chunk waiting for its DP) and its argument (err[10]).
__device__ __forceinline__ void report_timeout(int32_t* err, int site, int arg) {
    if (atomicCAS(err + 9, 0, site) == 0) atomicExch(err + 10, arg);
    atomicOr(err, ERR_TIMEOUT);
}
// Bounded wait for the copy of phase `parity`; false (error flag raised) on timeout.

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                                          int limit = kWaitSpins) {
    for (int i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    report_timeout(err, 1, (int)parity);
    return false;
}

// Rows of one warp's grid-stride sequence of 32-row batches: position k is
// row (b0 + (k/32)*wstride)*32 + k%32; positions [0, count) are valid rows.
struct WarpRows {
    int64_t b0, wstride, count;
    __device__ __forceinline__ void init(int64_t rows, int64_t warp, int64_t nwarps) {
        b0 = warp;
        wstride = nwarps;
        const int64_t nbatch = (rows + 31) / 32;
        if (b0 >= nbatch) {
            count = 0;
            return;
        }
        const int64_t nb = (nbatch - 1 - b0) / wstride + 1;   // batches of this warp
        const int64_t last = b0 + (nb - 1) * wstride;
        count = (nb - 1) * 32 + min((int64_t)32, rows - last * 32);
    }
    __device__ __forceinline__ int64_t row(int64_t k) const {
        return (b0 + (k >> 5) * wstride) * 32 + (k & 31);
    }
};

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}
__device__ __forceinline__ int smid() {
    int v;
    asm volatile("mov.u32 %0, %%smid;\n" : "=r"(v));
    return v;
}

// Trace record of task t: {kind | sample << 2, sm, start, end}, times in ns
// since k_prepare started (err[4..5] hold that origin).
__device__ __forceinline__ void trace_task(const Params& p, int t, int code, uint64_t t_start) {
    if (t >= p.trace_cap) return;
    const uint64_t origin = *reinterpret_cast<const uint64_t*>(p.err + 4);
    p.trace[t] = make_int4(code, smid(), (int)(t_start - origin), (int)(global_ns() - origin));
}

// Log-softmax partials of one row held as NV 16-byte vectors per lane
// (vector wl + 32 i of the row), for this lane's elements only: m = their
// maximum and s = sum of 2^(h log2 e - m log2 e) over them (m = -inf, s = 0
// for a lane without finite elements).  No cross-lane work: the partials of
// eight rows are merged together by lse_group8.  The maximum is folded over
// packed half2 (or float) words first and widened once; exponent arguments
// and the two partial sums (even and odd elements) use packed fp32x2 FMA/add.
template <typename Tin, int NV>
__device__ __forceinline__ void row_partial(const uint4* q, int nvec, int wl, float& m, float& s) {
    if constexpr (std::is_same<Tin, __half>::value) {
        __half2 m2 = __half2half2(__ushort_as_half((unsigned short)0xfc00u));   // -inf
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            if (wl + 32 * i < nvec) {
                const __half2* h = reinterpret_cast<const __half2*>(&q[i]);
                m2 = __hmax2(m2, __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3])));
            }
        }
        const float2 mf = __half22float2(m2);
        m = fmaxf(mf.x, mf.y);
    } else if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
        __nv_bfloat162 m2 = __bfloat162bfloat162(__ushort_as_bfloat16((unsigned short)0xff80u));
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            if (wl + 32 * i < nvec) {
                const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q[i]);
                m2 = __hmax2(m2, __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3])));
            }
        }
        const float2 mf = __bfloat1622float2(m2);
        m = fmaxf(mf.x, mf.y);
    } else {
        m = -INFINITY;
#pragma unroll
        for (int i = 0; i < NV; ++i)
            if (wl + 32 * i < nvec)
                m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(q[i].x), __uint_as_float(q[i].y)),
                                   fmaxf(__uint_as_float(q[i].z), __uint_as_float(q[i].w))));
    }
    float2 acc = make_float2(0.0f, 0.0f);
    const float mL = (m == -INFINITY) ? 0.0f : m * kLog2e;
    const float2 l2 = make_float2(kLog2e, kLog2e), c2 = make_float2(-mL, -mL);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        if (wl + 32 * i < nvec) {
            float2 f[4];
            if constexpr (std::is_same<Tin, __half>::value) {
                const __half2* h = reinterpret_cast<const __half2*>(&q[i]);
#pragma unroll
                for (int k = 0; k < 4; ++k) f[k] = __half22float2(h[k]);
            } else if constexpr (std::is_same<Tin, __nv_bfloat16>::value) {
                const uint32_t w[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    f[k] = make_float2(__uint_as_float(w[k] << 16),
                                       __uint_as_float(w[k] & 0xffff0000u));
            } else {
                f[0] = make_float2(__uint_as_float(q[i].x), __uint_as_float(q[i].y));
                f[1] = make_float2(__uint_as_float(q[i].z), __uint_as_float(q[i].w));
            }
            constexpr int NF = sizeof(Tin) == 2 ? 4 : 2;
#pragma unroll
            for (int k = 0; k < NF; ++k) {
                float2 t = __ffma2_rn(f[k], l2, c2);
                t.x = ex2(t.x);
                t.y = ex2(t.y);
                acc = __fadd2_rn(acc, t);
            }
        }
    }
    s = acc.x + acc.y;
}

// Merges the log-softmax partial (bm, bs) into (am, as): the result stands for
// max(am, bm) and the sum rescaled to it.  Bit-for-bit symmetric in its two
// operands (the larger maximum's sum plus the other sum times 2^-|d|), so the
// lanes of a butterfly all end with the same value.
__device__ __forceinline__ void lse_merge(float& am, float& as, float bm, float bs) {
    const float d = (bm - am) * kLog2e;
    const float e = ex2(-fabsf(d));
    const bool bigger = d > 0.0f;
    const float hi = bigger ? bs : as, lo = bigger ? as : bs;
    const bool skip = bm == -INFINITY;   // nothing to merge (also covers both -inf)
    as = skip ? as : fmaf(lo, e, hi);
    am = skip ? am : (bigger ? bm : am);
}

// Warp: merges every lane's partials (lm[j], ls[j]) of eight rows j = 0..7 by a
// transposing butterfly (9 merges and 18 shuffles per lane for all eight
// rows); on return lanes 4j..4j+3 hold row j's maximum M and sum S (relative
// to M).  A row's result depends only on its own partials, whatever rows
// share the group.
__device__ __forceinline__ void lse_group8(const float (&lm)[8], const float (&ls)[8], int wl,
                                           float& M, float& S) {
    constexpr unsigned F = 0xffffffffu;
    float am[4], as[4];
    const bool h16 = wl & 16;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        am[k] = h16 ? lm[4 + k] : lm[k];
        as[k] = h16 ? ls[4 + k] : ls[k];
        const float rm = __shfl_xor_sync(F, h16 ? lm[k] : lm[4 + k], 16);
        const float rs = __shfl_xor_sync(F, h16 ? ls[k] : ls[4 + k], 16);
        lse_merge(am[k], as[k], rm, rs);
    }
    float bm[2], bs[2];
    const bool h8 = wl & 8;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        bm[k] = h8 ? am[2 + k] : am[k];
        bs[k] = h8 ? as[2 + k] : as[k];
        const float rm = __shfl_xor_sync(F, h8 ? am[k] : am[2 + k], 8);
        const float rs = __shfl_xor_sync(F, h8 ? as[k] : as[2 + k], 8);
        lse_merge(bm[k], bs[k], rm, rs);
    }
    const bool h4 = wl & 4;
    M = h4 ? bm[1] : bm[0];
    S = h4 ? bs[1] : bs[0];
    {
        const float rm = __shfl_xor_sync(F, h4 ? bm[0] : bm[1], 4);
        const float rs = __shfl_xor_sync(F, h4 ? bs[0] : bs[1], 4);
        lse_merge(M, S, rm, rs);
    }
#pragma unroll
    for (int o = 2; o > 0; o >>= 1) {
        const float rm = __shfl_xor_sync(F, M, o), rs = __shfl_xor_sync(F, S, o);
        lse_merge(M, S, rm, rs);
    }
}

// ---------------------------------------------------------------- k_prepare
enum : int { TASK_ROW = 0, TASK_DP = 1, TASK_GRAD = 2 };

// Exclusive block-wide scan of one int64 per thread (all threads call it);
// `carry` (shared) accumulates across successive calls.
__device__ __forceinline__ int64_t block_scan_excl(int64_t n, int64_t* wsum, int64_t& carry) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int64_t x = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int64_t w = (lane < (int)(blockDim.x >> 5)) ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    const int64_t excl = carry + (wid ? wsum[wid - 1] : 0) + x - n;
    __syncthreads();
    if (tid == (int)blockDim.x - 1) carry = excl + n;
    __syncthreads();
    return excl;
}

// Appends the chunk tasks of `kind` for every sample in DP order (p.order),
// starting at task index t0, and returns how many it appended; chunks hold
// kTaskRows rows (the last one of a sample fewer).  The row pass also resets
// the per-sample scheduler counters.  A task record (32 bytes) holds all a
// CTA needs to start it: kind, sample, rows, the sample's lengths and first
// row, so starting a task takes one round of loads.
// The chunks of one sample are written by one warp, a chunk per lane.
__device__ int64_t append_chunks(const Params& p, int64_t t0, int kind, int64_t* wsum,
                                 int64_t& carry, int64_t* s_before, int* s_nch) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nwarps = blockDim.x >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < p.B; base += blockDim.x) {
        const int i = base + tid;
        int nch = 0;
        if (i < p.B) {
            const int b = p.order[i];
            const int64_t nrows = (int64_t)p.Tl[b] * (p.Ul[b] + 1);
            nch = (int)((nrows + kTaskRows - 1) / kTaskRows);
            if (kind == TASK_ROW) {
                p.rtasks[b] = nch;
                p.rdone[b] = 0;
                p.dpdone[b] = 0;
                p.dpclaim[b] = 0;
            }
        }
        s_before[tid] = block_scan_excl(nch, wsum, carry);   // chunks before position i
        s_nch[tid] = nch;
        __syncthreads();
        const int nb = min((int)blockDim.x, p.B - base);
        for (int j = wid; j < nb; j += nwarps) {
            const int ii = base + j;
            const int b = p.order[ii];
            const int T = p.Tl[b], U = p.Ul[b];
            const int64_t nrows = (int64_t)T * (U + 1);
            const int64_t o = __ldcg(p.off + b);
            for (int k = lane; k < s_nch[j]; k += 32) {
                const int r = k * kTaskRows;
                int4* rec = p.tasks + 2 * (t0 + s_before[j] + k);
                rec[0] = make_int4(kind | (b << 2), r, (int)min((int64_t)kTaskRows, nrows - r), T);
                rec[1] = make_int4(U, 0, (int)(uint32_t)o, (int)(o >> 32));
            }
        }
        __syncthreads();
    }
    // Every thread reads the total before the next call's thread 0 resets carry.
    const int64_t total = carry;
    __syncthreads();
    return total;
}

// Validation, offsets, DP order and task list, by one CTA (every thread);
// s_before / s_nch: shared scratch of blockDim.x entries each.
__device__ void prepare_block(const Params& p, int64_t* s_before, int* s_nch) {
    __shared__ int64_t wsum[32];
    __shared__ int64_t carry;
    __shared__ int errs;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        carry = 0;
        errs = 0;
        *reinterpret_cast<uint64_t*>(p.err + 4) = global_ns();   // trace origin
        p.err[8] = 0;   // CTAs of the persistent kernel that have finished
        p.err[9] = 0;   // first timeout site (diagnosis)
        p.err[10] = 0;
        p.err[13] = 0;    // next zero-fill chunk
        p.err[14] = -1;   // SMs of the longest recursion's two CTAs (zero-fill CTAs skip them)
        p.err[15] = -1;
        // Rows per sample slot of the padded layout (0: compact), for rnnt_grad_scale.
        p.err[12] = p.padded ? p.maxT * p.maxW : 0;
    }
    __syncthreads();
    for (int base = 0; base < p.B; base += blockDim.x) {
        const int b = base + tid;
        int64_t n = 0;
        if (b < p.B) {
            const int T = p.Tl[b], U = p.Ul[b];
            if (T < 1 || U < 0 || U > p.S || U + 1 > kMaxW || (int64_t)T * (U + 1) > INT32_MAX ||
                (p.padded && (T > p.maxT || U + 1 > p.maxW)))
                atomicOr(&errs, ERR_LENGTH);
            else n = (int64_t)T * (U + 1);
        }
        int64_t x = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int64_t w = (lane < (int)(blockDim.x >> 5)) ? wsum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int64_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int64_t excl = carry + (wid ? wsum[wid - 1] : 0) + x - n;
        if (b < p.B) p.off[b] = excl;
        __syncthreads();
        if (tid == (int)blockDim.x - 1) carry = excl + n;
        __syncthreads();
    }
    if (tid == 0) {
        p.off[p.B] = carry;
        if (!p.padded && carry != p.rows) atomicOr(&errs, ERR_ROWS);
    }
    // Labels: in range and not blank (warp-transducer blog 5.2).
    // Eight labels per thread per round, their loads issued together.
    const int64_t nt = (int64_t)p.B * p.S;
    for (int64_t i0 = tid; i0 < nt; i0 += 8 * (int64_t)blockDim.x) {
        int y[8];
        bool need[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int64_t i = i0 + (int64_t)k * blockDim.x;
            need[k] = false;
            y[k] = 0;
            if (i < nt) {
                const int b = (int)(i / p.S), u = (int)(i % p.S);
                const int U = __ldg(p.Ul + b);
                need[k] = U >= 0 && U <= p.S && u < U;
                if (need[k]) y[k] = __ldg(p.targets + i);
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (need[k] && (y[k] < 0 || y[k] >= p.V || y[k] == p.blank)) atomicOr(&errs, ERR_TARGET);
            for (int i = 0; i < p.K; ++i)   // a big blank is never a label
                if (need[k] && y[k] == p.bb_id[i]) atomicOr(&errs, ERR_TARGET);
        }
    }
    // Longest DP first: key (T+U, area), ties by index.  O(B^2) rank sort.
    for (int b = tid; b < p.B; b += blockDim.x) {
        if (p.B > 8192) { p.order[b] = b; continue; }
        const int Tb = p.Tl[b], Ub = p.Ul[b];
        const int64_t kb = ((int64_t)(Tb + Ub) << 32) + (int64_t)Tb * (Ub + 1);
        int rank = 0;
        for (int j = 0; j < p.B; ++j) {
            const int Tj = p.Tl[j], Uj = p.Ul[j];
            const int64_t kj = ((int64_t)(Tj + Uj) << 32) + (int64_t)Tj * (Uj + 1);
            rank += (kj > kb) || (kj == kb && j < b);
        }
        p.order[rank] = b;
    }
    __syncthreads();
    // Task queue of the persistent kernel: the row chunks of every sample in DP
    // order, then the gradient chunks in the same order.  DP tasks are taken by
    // ticket (err[3]) in the same sample order.
    if (errs == 0 && p.build_tasks) {
        const int64_t nrow = append_chunks(p, 0, TASK_ROW, wsum, carry, s_before, s_nch);
        const int64_t ngrad = append_chunks(p, nrow, TASK_GRAD, wsum, carry, s_before, s_nch);
        if (tid == 0) {
            p.err[1] = 0;                          // next task
            p.err[2] = (int)(nrow + ngrad);        // task count
            p.err[3] = 0;                          // next DP ticket
        }
    }
    __syncthreads();
    if (tid == 0) *p.err = errs;
}

__global__ void __launch_bounds__(1024) k_prepare(Params p) {
    __shared__ int64_t s_before[1024];
    __shared__ int s_nch[1024];
    prepare_block(p, s_before, s_nch);
}

// ---------------------------------------------------------------- row pass
// G-lane groups reduce row statistics; every warp owns batches of 32
// consecutive rows and, once a batch is reduced, finishes it with one row per
// lane (sample lookup, label, transition probabilities, stores), so the
// scalar per-row work costs one warp instruction per 32 rows.

// One row per lane: log2 of the softmax denominator in row order, and the
// node's two transition probabilities at its node index.  A blank from the
// last frame before every label is out, and a label at u = U, have
// probability 0 (the lattice has no such arc).
template <typename Tin>
__device__ __forceinline__ void row_finish_at(const Params& p, int64_t r, float M, float s,
                                              float hb, float hy, int t, int u, int T, int U,
                                              int64_t o) {
    if (p.fused) {
        const float lse2v = fmaf(M, kLog2e, lg2(s));
        p.lse2[r] = lse2v;
        if (!(lse2v < INFINITY)) atomicOr(p.err, ERR_NONFINITE);   // NaN or +inf logits
    } else {
        p.lse2[r] = 0.0f;
        if (!(hb < INFINITY) || !(hy < INFINITY)) atomicOr(p.err, ERR_NONFINITE);
    }
    float bm = 0.0f, ym = 0.0f;
    int be = kZeroExp, ye = kZeroExp;
    if (!(t == T - 1 && u < U)) xf_prob(hb, M, s, bm, be);
    if (u < U) xf_prob(hy, M, s, ym, ye);
    p.edge[o + node_index(t, u, T, U)] =
        make_int4(__float_as_int(bm), be + kEdgeBias, __float_as_int(ym), ye + kEdgeBias);
}

// Row r with its sample looked up: the blank and label logits are read from
// global memory.
template <typename Tin>
__device__ __forceinline__ void row_finish(const Params& p, int64_t r, float M, float s) {
    using E = Elt<Tin>;
    const int b = find_sample(p.off, p.B, r);
    const int T = __ldg(p.Tl + b), U = __ldg(p.Ul + b), W = U + 1;
    const int64_t o = __ldcg(p.off + b);
    const Tin* row = static_cast<const Tin*>(p.logits) + lrow_s(p, r, b, o, W) * (int64_t)p.V;
    const unsigned rr = (unsigned)(r - o);
    const int t = (int)(rr / (unsigned)W), u = (int)(rr - (unsigned)t * W);
    const float hb = E::get(row, p.blank);
    const float hy = (u < U) ? E::get(row, __ldg(p.targets + (int64_t)b * p.S + u)) : 0.0f;
    row_finish_at<Tin>(p, r, M, s, hb, hy, t, u, T, U, o);
    // Multi-blank: every big blank's probability at this node.
    const int64_t nd = o + node_index(t, u, T, U);
    for (int i = 0; i < p.K; ++i) {
        float m;
        int e;
        xf_prob(E::get(row, p.bb_id[i]), M, s, m, e);
        p.pbb[(int64_t)i * p.rows + nd] = make_int2(__float_as_int(m), e + kEdgeBias);
    }
}

// Group results (same in every lane of group g) for row it*NG+g of the batch
// are handed to the lane with that index.
template <int G>
__device__ __forceinline__ void hand_over(int it, int wl, float M, float s, float& myM,
                                          float& mys) {
    constexpr int NG = 32 / G;
    const float vM = __shfl_sync(0xffffffffu, M, (wl % NG) * G);
    const float vs = __shfl_sync(0xffffffffu, s, (wl % NG) * G);
    if (wl / NG == it) {
        myM = vM;
        mys = vs;
    }
}

// Rows held in registers: NV 16-byte vectors per lane, the next row's
// vectors loaded before the current one is reduced.
template <typename Tin, int G, int NV>
__global__ void __launch_bounds__(256) k_row_regs(Params p) {
    if (*p.err) return;
    using E = Elt<Tin>;
    constexpr int EPV = E::kPerVec, NG = 32 / G;
    const Tin* X = static_cast<const Tin*>(p.logits);
    const int V = p.V, nvec = V / EPV;
    const int wl = threadIdx.x & 31, lane = wl & (G - 1), grp = wl / G;
    const unsigned gm = group_mask<G>();
    const int64_t nbatch = (nodes(p) + 31) / 32;
    const int64_t wstride = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t bt = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; bt < nbatch;
         bt += wstride) {
        const int64_t r0 = bt * 32;
        const int nrows = (int)min((int64_t)32, nodes(p) - r0);
        float myM = 0.0f, mys = 0.0f;
        uint4 cur[NV];
        if (grp < nrows) {
            const uint4* rv = reinterpret_cast<const uint4*>(X + lrow(p, r0 + grp) * (int64_t)V);
#pragma unroll
            for (int k = 0; k < NV; ++k)
                if (lane + k * G < nvec) cur[k] = __ldg(rv + lane + k * G);
        }
        for (int it = 0; it < G; ++it) {
            const int ri = it * NG + grp;
            uint4 nxt[NV];
            if (ri + NG < nrows) {
                const uint4* rv =
                    reinterpret_cast<const uint4*>(X + lrow(p, r0 + ri + NG) * (int64_t)V);
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    if (lane + k * G < nvec) nxt[k] = __ldg(rv + lane + k * G);
            }
            float M = -INFINITY, s = 0.0f;
            if (ri < nrows) {
#pragma unroll
                for (int k = 0; k < NV; ++k)
                    if (lane + k * G < nvec) M = fmaxf(M, E::vmax(cur[k]));
                M = group_max<G>(M, gm);
                if (M != -INFINITY) {
                    const float ML = M * kLog2e;
#pragma unroll
                    for (int k = 0; k < NV; ++k) {
                        if (lane + k * G < nvec) {
                            float x[EPV];
                            E::unpack(cur[k], x);
#pragma unroll
                            for (int e = 0; e < EPV; ++e) s += ex2(fmaf(x[e], kLog2e, -ML));
                        }
                    }
                }
                s = group_sum<G>(s, gm);
            }
            hand_over<G>(it, wl, M, s, myM, mys);
#pragma unroll
            for (int k = 0; k < NV; ++k) cur[k] = nxt[k];
        }
        if (wl < nrows) row_finish<Tin>(p, r0 + wl, myM, mys);
    }
}

// Rows of up to 32*NV 16-byte vectors staged through shared memory by TMA:
// a warp streams its row sequence with kStages-1 rows in flight.
template <typename Tin, int NV>
__global__ void __launch_bounds__(256) k_row_tma(Params p) {
    if (*p.err) return;
    using E = Elt<Tin>;
    constexpr int EPV = E::kPerVec;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int nw = blockDim.x >> 5, wid = threadIdx.x >> 5, wl = threadIdx.x & 31;
    const int sb = p.stage_bytes;
    unsigned char* buf = smem_raw + (size_t)wid * kStages * sb;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (size_t)nw * kStages * sb) + wid * kStages;
    if (wl == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const Tin* X = static_cast<const Tin*>(p.logits);
    const int V = p.V, nvec = V / EPV;
    const uint32_t rb = (uint32_t)V * sizeof(Tin);
    WarpRows seq;
    seq.init(nodes(p), (int64_t)blockIdx.x * nw + wid, (int64_t)gridDim.x * nw);
    if (wl == 0)
        for (int64_t k = 0; k < min((int64_t)kStages, seq.count); ++k)
            tma_row_load(buf + (k % kStages) * sb, X + lrow(p, seq.row(k)) * (int64_t)V, rb,
                         &bars[k % kStages]);
    // Groups of 8 sequence positions (8-aligned, so inside one 32-row batch):
    // per-lane partials of each row, then one butterfly merge per group.
    float myM = 0.0f, mys = 0.0f;
    int64_t kfail = -1;
    for (int64_t k0 = 0; k0 < seq.count; k0 += 8) {
        float lm[8], ls[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            lm[j] = -INFINITY;
            ls[j] = 0.0f;
            const int64_t k = k0 + j;
            if (kfail < 0 && k < seq.count) {
                const int st = (int)(k % kStages);
                if (!mbar_wait(&bars[st], (uint32_t)((k / kStages) & 1), p.err)) {
                    kfail = k;
                } else {
                    const uint4* rv = reinterpret_cast<const uint4*>(buf + st * sb);
                    uint4 q[NV];
#pragma unroll
                    for (int i = 0; i < NV; ++i)
                        if (wl + 32 * i < nvec) q[i] = rv[wl + 32 * i];
                    __syncwarp();
                    if (wl == 0 && k + kStages < seq.count) {   // refill this stage
                        fence_proxy_async();
                        tma_row_load(buf + st * sb, X + lrow(p, seq.row(k + kStages)) * (int64_t)V, rb,
                                     &bars[st]);
                    }
                    row_partial<Tin, NV>(q, nvec, wl, lm[j], ls[j]);
                }
            }
        }
        if (kfail >= 0) break;
        float M, S;
        lse_group8(lm, ls, wl, M, S);
        const float vM = __shfl_sync(0xffffffffu, M, 4 * (wl & 7));
        const float vS = __shfl_sync(0xffffffffu, S, 4 * (wl & 7));
        if ((wl & 24) == (int)(k0 & 31)) {
            myM = vM;
            mys = vS;
        }
        const int64_t kl = min(k0 + 7, seq.count - 1);
        const int it = (int)(kl & 31);
        if (it == 31 || kl == seq.count - 1) {
            if (wl <= it) row_finish<Tin>(p, seq.row(kl - it + wl), myM, mys);
        }
    }
    // After a timeout, wait (bounded) for the copies still in flight before exiting.
    if (kfail >= 0)
        for (int64_t q = kfail; q < min(kfail + kStages, seq.count); ++q)
            mbar_wait(&bars[q % kStages], (uint32_t)((q / kStages) & 1), p.err);
}

// Long rows (or rows not 16-byte aligned): streaming max/sum with rescale.
template <typename Tin, int G, bool VEC>
__device__ __forceinline__ void row_stats_stream(const Tin* row, int V, int lane, unsigned gm,
                                                 float& Mo, float& so) {
    using E = Elt<Tin>;
    float m = -INFINITY, s = 0.0f;
    if (VEC) {
        constexpr int EPV = E::kPerVec, UNR = 4;
        const uint4* rv = reinterpret_cast<const uint4*>(row);
        const int nvec = V / EPV;
        for (int v0 = lane; v0 < nvec; v0 += G * UNR) {
            float x[UNR * EPV];
#pragma unroll
            for (int k = 0; k < UNR; ++k) {
                const int vi = v0 + k * G;
                if (vi < nvec) {
                    E::unpack(__ldg(rv + vi), x + k * EPV);
                } else {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) x[k * EPV + e] = -INFINITY;
                }
            }
            float cm = x[0];
#pragma unroll
            for (int e = 1; e < UNR * EPV; ++e) cm = fmaxf(cm, x[e]);
            const float nm = fmaxf(m, cm);
            if (nm != -INFINITY) {
                if (nm != m) s *= ex2((m - nm) * kLog2e);
                const float nmL = nm * kLog2e;
#pragma unroll
                for (int e = 0; e < UNR * EPV; ++e) s += ex2(fmaf(x[e], kLog2e, -nmL));
                m = nm;
            } else {   // nothing but -inf and NaN so far: a NaN still reaches the sum
#pragma unroll
                for (int e = 0; e < UNR * EPV; ++e)
                    if (x[e] != x[e]) s = x[e];
            }
        }
    } else {
        constexpr int UNR = 8;
        for (int k0 = lane; k0 < V; k0 += G * UNR) {
            float x[UNR];
#pragma unroll
            for (int k = 0; k < UNR; ++k) {
                const int kk = k0 + k * G;
                x[k] = (kk < V) ? E::get(row, kk) : -INFINITY;
            }
            float cm = x[0];
#pragma unroll
            for (int e = 1; e < UNR; ++e) cm = fmaxf(cm, x[e]);
            const float nm = fmaxf(m, cm);
            if (nm != -INFINITY) {
                if (nm != m) s *= ex2((m - nm) * kLog2e);
                const float nmL = nm * kLog2e;
#pragma unroll
                for (int e = 0; e < UNR; ++e) s += ex2(fmaf(x[e], kLog2e, -nmL));
                m = nm;
            } else {   // nothing but -inf and NaN so far: a NaN still reaches the sum
#pragma unroll
                for (int e = 0; e < UNR; ++e)
                    if (x[e] != x[e]) s = x[e];
            }
        }
    }
    const float M = group_max<G>(m, gm);
    s = (M == -INFINITY) ? 0.0f : s * ex2((m - M) * kLog2e);
    Mo = M;
    so = group_sum<G>(s, gm);
}

// ---- Short rows that are not 16-byte vectors (compact layout) ----
// Up to kFlatRowBytes bytes per row.  A warp stages up to 32 consecutive
// rows into shared memory: coalesced 16-byte loads of the 16-byte aligned
// span that holds them (its first chunk may start inside the previous row;
// the bytes past its last full chunk are loaded element by element, so
// nothing past the tensor is read); lane l then reduces row l there, the
// maximum and then the sum of 2^((x - max) log2 e) in element order.  Both
// schedules use these functions, so they give the same bits.
constexpr int kFlatRowBytes = 256;
__host__ __device__ inline size_t flat_warp_bytes(int V, int es) {
    return (size_t)32 * V * es + 32;
}
// (The padded layout reduces such rows the same way, each lane reading its
// row from global memory: padded and compact calls agree bit for bit.)
__host__ __device__ inline bool flat_rows(int V, int es, int fused) {
    return fused && ((size_t)V * es) % 16 != 0 && (size_t)V * es <= kFlatRowBytes;
}

template <typename Tin>
__device__ __forceinline__ const Tin* flat_stage(const Tin* X, int64_t r0, int n, int V,
                                                 unsigned char* sbuf, int lane) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(X + r0 * (int64_t)V);
    const uintptr_t e = reinterpret_cast<uintptr_t>(X + (r0 + n) * (int64_t)V);
    const uintptr_t a0 = a & ~uintptr_t(15), e0 = e & ~uintptr_t(15);
    const int nv = (int)((e0 - a0) / 16);
    const uint4* src = reinterpret_cast<const uint4*>(a0);
    uint4* dst = reinterpret_cast<uint4*>(sbuf);
    for (int i = lane; i < nv; i += 32) dst[i] = __ldcs(src + i);
    const int nt = (int)((e - e0) / sizeof(Tin));
    if (lane < nt)
        reinterpret_cast<Tin*>(sbuf + (e0 - a0))[lane] = reinterpret_cast<const Tin*>(e0)[lane];
    __syncwarp();
    return reinterpret_cast<const Tin*>(sbuf + (a - a0));
}

template <typename Tin>
__device__ __forceinline__ void flat_row_stats(const Tin* row, int V, float& M, float& s) {
    using E = Elt<Tin>;
    float m = -INFINITY;
    for (int k = 0; k < V; ++k) m = fmaxf(m, E::to_f(row[k]));
    const float mL = m == -INFINITY ? 0.0f : m * kLog2e;
    float acc = 0.0f;   // a NaN element makes it NaN (fmaxf above skips it)
    for (int k = 0; k < V; ++k) acc += ex2(fmaf(E::to_f(row[k]), kLog2e, -mL));
    M = m;
    s = acc;
}

// Gradient of n <= 32 consecutive compact rows from r0 (log-softmax on) in
// flat element order: lane l takes elements l, l + 32, ... of the rows'
// contiguous span, four at a time with their loads issued together; rec(i)
// gives row i's record (called by every lane, same trip count).  Rows of exact
// zeros are not read.
template <typename Tin, typename Rec>
__device__ __forceinline__ void flat_grad(const Params& p, int64_t r0, int n, int lane, Rec rec) {
    using E = Elt<Tin>;
    constexpr int UF = 4;
    const int V = p.V;
    const Tin* X = static_cast<const Tin*>(p.logits) + r0 * (int64_t)V;
    Tin* Y = static_cast<Tin*>(p.grad) + r0 * (int64_t)V;
    const float invV = 1.0f / (float)V;   // (f + 1/2) / V floors exactly for f < 32 V <= 2^13
    const float cl = p.clamp * p.scale;
    const bool clip = p.clamp < INFINITY;
    const int nel = n * V;
    for (int f0 = 0; f0 < nel; f0 += 32 * UF) {
        float x[UF];
        float4 rc[UF];
        int kk[UF];
#pragma unroll
        for (int u = 0; u < UF; ++u) {
            const int f = f0 + 32 * u + lane;
            const int rw = f < nel ? (int)(((float)f + 0.5f) * invV) : 0;
            kk[u] = f - rw * V;
            rc[u] = rec(rw);
            x[u] = (f < nel && rc[u].x != -INFINITY) ? E::to_f(__ldcs(X + f)) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < UF; ++u) {
            const int f = f0 + 32 * u + lane;
            if (f >= nel) break;
            float gv = rc[u].x != -INFINITY ? ex2(fmaf(x[u], kLog2e, rc[u].x)) : 0.0f;
            if (kk[u] == p.blank) gv -= rc[u].y;
            if (kk[u] == __float_as_int(rc[u].w)) gv -= rc[u].z;
            if (clip) gv = fminf(fmaxf(gv, -cl), cl);
            __stcs(Y + f, E::from_f(gv));
        }
    }
}

// Per-stage row pass for such rows: a warp per 32-row chunk (grid-stride).
template <typename Tin>
__global__ void __launch_bounds__(256) k_row_flat(Params p) {
    if (*p.err) return;
    extern __shared__ __align__(16) unsigned char flat_smem[];
    const int wl = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned char* sbuf = flat_smem + (size_t)wid * flat_warp_bytes(p.V, sizeof(Tin));
    const Tin* X = static_cast<const Tin*>(p.logits);
    const int64_t nr = nodes(p), nbatch = (nr + 31) / 32;
    const int64_t wstride = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t bt = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; bt < nbatch;
         bt += wstride) {
        const int64_t r0 = bt * 32;
        const int n = (int)min((int64_t)32, nr - r0);
        float M = 0.0f, s = 0.0f;
        if (p.padded) {
            if (wl < n) flat_row_stats<Tin>(X + lrow(p, r0 + wl) * (int64_t)p.V, p.V, M, s);
        } else {
            const Tin* rows = flat_stage<Tin>(X, r0, n, p.V, sbuf, wl);
            if (wl < n) flat_row_stats<Tin>(rows + (int64_t)wl * p.V, p.V, M, s);
            __syncwarp();   // the buffer is reused by the next chunk
        }
        if (wl < n) row_finish<Tin>(p, r0 + wl, M, s);
    }
}

template <typename Tin, int G, bool VEC>
__global__ void __launch_bounds__(256) k_row_stream(Params p) {
    if (*p.err) return;
    constexpr int NG = 32 / G;
    const Tin* X = static_cast<const Tin*>(p.logits);
    const int wl = threadIdx.x & 31, lane = wl & (G - 1), grp = wl / G;
    const unsigned gm = group_mask<G>();
    const int64_t nbatch = (nodes(p) + 31) / 32;
    const int64_t wstride = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t bt = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; bt < nbatch;
         bt += wstride) {
        const int64_t r0 = bt * 32;
        const int nrows = (int)min((int64_t)32, nodes(p) - r0);
        float myM = 0.0f, mys = 0.0f;
        for (int it = 0; it < G; ++it) {
            const int ri = it * NG + grp;
            float M = -INFINITY, s = 0.0f;
            if (ri < nrows)
                row_stats_stream<Tin, G, VEC>(X + lrow(p, r0 + ri) * (int64_t)p.V, p.V, lane, gm,
                                              M, s);
            hand_over<G>(it, wl, M, s, myM, mys);
        }
        if (wl < nrows) row_finish<Tin>(p, r0 + wl, myM, mys);
    }
}

// In-kernel log-softmax off: the rows already hold log-probs; read 2 elements.

// ---------------------------------------------------------------- DP
// One CTA per sample (8 warps).  Per direction, nwd compute warps (at most
// 4; W = U+1 lattice columns) each own a contiguous block of 32*J columns,
// J = ceil(W/(32*nwd)) <= 8; lane l holds columns u0 + 32*j + l.  The
// neighbouring column comes from the next lane by shuffle, or at a block
// edge from the neighbouring warp through shared memory with one named
// barrier per anti-diagonal (1: alpha, 2: beta).  Alpha and beta warps
// interleave (even / odd warp ids).  Each compute warp prefetches its nodes'
// transition records with zero-filling cp.async into a ring of R diagonals
// (prefetch distance R-2).  Per-diagonal bookkeeping is kept small: the
// diagonal's base index comes by shuffle from a 32-diagonal window, and
// each lane keeps per-column pointers.
template <int J> struct Ring;
template <> struct Ring<1> { static constexpr int R = 16; };
template <> struct Ring<2> { static constexpr int R = 12; };
constexpr int kDpWarps = 4;         // compute warps per direction, at most (both directions on one CTA)
constexpr int kDpWarpsStaged = 4;   // the same for the per-stage DP (one direction per CTA)

// The DP's ring copies, waits and ring reads are all volatile asm without a
// "memory" clobber: volatile asm statements keep their relative order (copy,
// wait, read), while the compiler stays free to move the recursion's
// arithmetic and its global stores around them.
__device__ __forceinline__ void cp16z(void* smem, const void* gmem, bool valid) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(sa), "l"(gmem),
                 "r"(valid ? 16 : 0));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }
__device__ __forceinline__ int4 lds128(const int4* ptr) {
    int4 v;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"((unsigned)__cvta_generic_to_shared(ptr)));
    return v;
}
__device__ __forceinline__ void sts64(float2* ptr, float2 v) {
    asm volatile("st.shared.v2.f32 [%0], {%1, %2};\n" ::"r"((unsigned)__cvta_generic_to_shared(ptr)),
                 "f"(v.x), "f"(v.y));
}
__device__ __forceinline__ float2 lds64(const float2* ptr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];\n"
                 : "=f"(v.x), "=f"(v.y)
                 : "r"((unsigned)__cvta_generic_to_shared(ptr)));
    return v;
}
// Orders the volatile shared-memory exchange (sts64 before, lds64 after).
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads));
}

struct Samp {
    int b, T, U, W, D;
    int64_t off;
};

// The node in column u on diagonal d is at index base(d) - u with
// base(d) = N(d) - max(0, d-U) + d (N(d) = nodes before diagonal d).
__device__ __forceinline__ int diag_base(const Samp& c, int d) {
    return (int)(diag_start(d, c.T, c.W) - max(0, d - c.U) + d);
}

// Diagonal bases for a window of 32 consecutive diagonals, one per lane
// (lane l: diagonal first + dir*l); a diagonal's base is then one shuffle.
struct BaseWin {
    int first, dir, mine;
    __device__ __forceinline__ void load(const Samp& c, int f, int dr, int lane) {
        first = f;
        dir = dr;
        const int d = f + dr * lane;
        mine = (d >= 0 && d < c.D) ? diag_base(c, d) : 0;
    }
    // Base of diagonal d (warp-uniform d inside or just past the window).
    __device__ __forceinline__ int get(const Samp& c, int d, int lane) {
        int k = (d - first) * dir;
        if (k >= 32) {   // warp-uniform refill
            load(c, first + 32 * dir, dir, lane);
            k -= 32;
        }
        return __shfl_sync(0xffffffffu, mine, k);
    }
};

template <int J>
struct Lanes {
    int u[J];          // this lane's columns u0 + 32j + lane
    int Tl[J];         // T if the column exists (u <= U), else 0
    const int4* e[J];  // edge records of this column: e[j][base(d)] is node (d-u, u)
    int2* o[J];        // output (alpha or beta) of this column, same indexing
};

template <int J>
__device__ __forceinline__ void lanes_init(const Samp& c, int u0, int lane, const int4* edge_s,
                                           int2* out_s, Lanes<J>& L) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
        L.u[j] = u0 + 32 * j + lane;
        L.Tl[j] = L.u[j] <= c.U ? c.T : 0;
        L.e[j] = edge_s - L.u[j];
        L.o[j] = out_s - L.u[j];
    }
}

// Zero-filling copies of the transition records of diagonal e (base be)
// into a ring slot; records of missing nodes read as probability 0.
template <int J>
__device__ __forceinline__ void ring_issue(int4* slot, int e, int be, const Lanes<J>& L) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const bool ok = (unsigned)(e - L.u[j]) < (unsigned)L.Tl[j];
        cp16z(slot + j * 32, ok ? L.e[j] + be : L.e[j] + L.u[j], ok);
    }
}

template <int J>
__device__ __forceinline__ void store_diag(int d, int bd, const Lanes<J>& L, const float* m,
                                           const int* e) {
#pragma unroll
    for (int j = 0; j < J; ++j)
        if ((unsigned)(d - L.u[j]) < (unsigned)L.Tl[j])
            L.o[j][bd] = make_int2(__float_as_int(m[j]), e[j]);
}

// Forward variable: alpha(t,u) = alpha(t-1,u) p_blank(t-1,u) + alpha(t,u-1) p_label(t,u-1).
// xch: [2][kDpWarpsStaged] (m, e) of the label arc leaving each warp's last column.
template <int J, int R = Ring<J>::R>
__device__ void dp_alpha(const Params& p, const Samp& c, int u0, int w, int nwd, int4* ring,
                         float2* xch) {
    constexpr int PF = R - 2;
    const int lane = threadIdx.x & 31, nthreads = nwd * 32;
    Lanes<J> L;
    lanes_init<J>(c, u0, lane, p.edge + c.off, p.alpha + c.off, L);
    float am[J];
    int ae[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        am[j] = L.u[j] == 0 ? 1.0f : 0.0f;
        ae[j] = L.u[j] == 0 ? 0 : kZeroExp;
    }
    store_diag<J>(0, 0, L, am, ae);   // alpha(0,0) = 1 (base(0) = 0)
    int4* const rl = ring + lane;
    BaseWin wi, ws;
    wi.load(c, 0, 1, lane);
    ws.load(c, 1, 1, lane);
    // Diagonal e's records feed diagonal e+1; prefetch PF diagonals.
    int e = 0, si = 0;
    for (; e < PF; ++e) {
        const int be = wi.get(c, e, lane);
        if (e < c.D) ring_issue<J>(rl + si * (J * 32), e, be, L);
        cp_commit();
        si = si + 1 == R ? 0 : si + 1;
    }
    int so = 0;
    auto step = [&](int d, auto norm) {
        {
            const int be = wi.get(c, e, lane);
            if (e < c.D) ring_issue<J>(rl + si * (J * 32), e, be, L);
            cp_commit();
            ++e;
            si = si + 1 == R ? 0 : si + 1;
        }
        cp_wait<PF>();
        const int4* sp = rl + so * (J * 32);
        so = so + 1 == R ? 0 : so + 1;
        float bm[J], ym[J];
        int be[J], ye[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int4 ed = lds128(sp + j * 32);
            xf_mul(am[j], ae[j], __int_as_float(ed.x), ed.y - kEdgeBias, bm[j], be[j]);
            xf_mul(am[j], ae[j], __int_as_float(ed.z), ed.w - kEdgeBias, ym[j], ye[j]);
        }
        float edge_m = 0.0f;
        int edge_e = kZeroExp;
        if (nwd > 1) {
            if (lane == 31)
                sts64(xch + (d & 1) * kDpWarpsStaged + w, make_float2(ym[J - 1], __int_as_float(ye[J - 1])));
            named_barrier(1, nthreads);
            const float2 v = lds64(xch + (d & 1) * kDpWarpsStaged + max(w - 1, 0));
            if (w > 0) {
                edge_m = v.x;
                edge_e = __float_as_int(v.y);
            }
        }
        float sm[J];
        int se[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            sm[j] = __shfl_sync(0xffffffffu, ym[j], (lane + 31) & 31);
            se[j] = __shfl_sync(0xffffffffu, ye[j], (lane + 31) & 31);
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const float nm = lane ? sm[j] : (j ? sm[j - 1] : edge_m);
            const int ne = lane ? se[j] : (j ? se[j - 1] : edge_e);
            xf_add<decltype(norm)::value>(bm[j], be[j], nm, ne, am[j], ae[j]);
        }
        store_diag<J>(d, ws.get(c, d, lane), L, am, ae);
    };
    int d = 1;
    for (; d + 1 < c.D; d += 2) {
        step(d, std::false_type());
        step(d + 1, std::true_type());
    }
    if (d < c.D) step(d, std::false_type());
    // P(y|x) = alpha(T-1,U) p_blank(T-1,U): the terminal blank (diagonal D-1).
    cp_wait<0>();
    const int4* sp = rl + so * (J * 32);
#pragma unroll
    for (int j = 0; j < J; ++j) {
        if (L.u[j] == c.U) {
            const int4 ed = lds128(sp + j * 32);
            float m;
            int x;
            xf_mul(am[j], ae[j], __int_as_float(ed.x), ed.y - kEdgeBias, m, x);
            xf_norm(m, x);
            p.pm[c.b] = m;
            p.pe[c.b] = x;
            const double ll2 = (double)x + log2((double)m);
            p.lossa[c.b] = -ll2 * kLn2d;
            p.loss[c.b] = (float)(-ll2 * kLn2d);
        }
    }
}

// Backward variable: beta(t,u) = beta(t+1,u) p_blank(t,u) + beta(t,u+1) p_label(t,u),
// started from a virtual node after the terminal blank with beta = 1.
// xch: [2][kDpWarpsStaged] (m, e) of each warp's first column on the previous diagonal.
template <int J, int R = Ring<J>::R>
__device__ void dp_beta(const Params& p, const Samp& c, int u0, int w, int nwd, int4* ring,
                        float2* xch) {
    constexpr int PF = R - 2;
    const int lane = threadIdx.x & 31, nthreads = nwd * 32;
    Lanes<J> L;
    lanes_init<J>(c, u0, lane, p.edge + c.off, p.beta + c.off, L);
    float vm[J];
    int ve[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        vm[j] = L.u[j] == c.U ? 1.0f : 0.0f;
        ve[j] = L.u[j] == c.U ? 0 : kZeroExp;
    }
    int4* const rl = ring + lane;
    BaseWin wi, ws;
    wi.load(c, c.D - 1, -1, lane);
    ws.load(c, c.D - 1, -1, lane);
    int e = c.D - 1, si = 0;
    for (int k = 0; k < PF; ++k, --e) {
        const int be = wi.get(c, e, lane);
        if (e >= 0) ring_issue<J>(rl + si * (J * 32), e, be, L);
        cp_commit();
        si = si + 1 == R ? 0 : si + 1;
    }
    int so = 0;
    auto step = [&](int d, auto norm) {
        {
            const int be = wi.get(c, e, lane);
            if (e >= 0) ring_issue<J>(rl + si * (J * 32), e, be, L);
            cp_commit();
            --e;
            si = si + 1 == R ? 0 : si + 1;
        }
        cp_wait<PF>();
        const int4* sd = rl + so * (J * 32);
        so = so + 1 == R ? 0 : so + 1;
        float edge_m = 0.0f;
        int edge_e = kZeroExp;
        if (nwd > 1) {
            if (lane == 0) sts64(xch + (d & 1) * kDpWarpsStaged + w, make_float2(vm[0], __int_as_float(ve[0])));
            named_barrier(2, nthreads);
            const float2 v = lds64(xch + (d & 1) * kDpWarpsStaged + min(w + 1, nwd - 1));
            if (w + 1 < nwd) {
                edge_m = v.x;
                edge_e = __float_as_int(v.y);
            }
        }
        float sm[J];
        int se[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            sm[j] = __shfl_sync(0xffffffffu, vm[j], (lane + 1) & 31);
            se[j] = __shfl_sync(0xffffffffu, ve[j], (lane + 1) & 31);
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int4 ed = lds128(sd + j * 32);
            const float nm = (lane < 31) ? sm[j] : (j + 1 < J ? sm[j + 1] : edge_m);
            const int ne = (lane < 31) ? se[j] : (j + 1 < J ? se[j + 1] : edge_e);
            float bm, ym;
            int be, ye;
            xf_mul(vm[j], ve[j], __int_as_float(ed.x), ed.y - kEdgeBias, bm, be);
            xf_mul(nm, ne, __int_as_float(ed.z), ed.w - kEdgeBias, ym, ye);
            xf_add<decltype(norm)::value>(bm, be, ym, ye, vm[j], ve[j]);
        }
        store_diag<J>(d, ws.get(c, d, lane), L, vm, ve);
    };
    int d = c.D - 1;
    for (; d >= 1; d -= 2) {
        step(d, std::false_type());
        step(d - 1, std::true_type());
    }
    if (d == 0) step(0, std::true_type());
    cp_wait<0>();
    if (u0 == 0 && lane == 0) p.lossb[c.b] = -((double)ve[0] + log2((double)vm[0])) * kLn2d;
}

// ---- DP over a table of diagonal bases (lattices with T+U <= kTabMax) ----
// The same recursions with branch-free steps: every step issues the copy of
// a future diagonal, waits for the next diagonal's records and loads them
// one step ahead, so the only latency left inside a step is the
// multiply -> shuffle -> add chain.  Warps of one direction are skewed by
// kSkew diagonals (warp w of alpha works on diagonal e at step e + kSkew*w;
// mirrored for beta), so a value crossing from one warp to the next was
// written at least kSkew steps before it is read, and one named barrier per
// kSkew steps orders the exchange.  Diagonal bases come from a shared table
// filled once per sample.
constexpr int kTabMax = 2048;   // table entries (diagonals)
constexpr int kSkew = 4;        // steps between barriers = skew between warps
constexpr int kXch = 16;        // exchange ring per warp (>= 2*kSkew + 2, a power of two)

template <int N>
__device__ __forceinline__ void cp_wait_mem() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
__device__ __forceinline__ void named_barrier_mem(int id, int threads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

// Copies of diagonal e's records (base be) into a ring slot; `live` false
// (e past the lattice) issues zero-filling copies that read nothing.
template <int J>
__device__ __forceinline__ void ring_issue_t(int4* slot, int e, int be, const Lanes<J>& L,
                                             bool live) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const bool ok = live && (unsigned)(e - L.u[j]) < (unsigned)L.Tl[j];
        cp16z(slot + j * 32, L.e[j] + (ok ? be : L.u[j]), ok);
    }
}

template <int R>
__device__ __forceinline__ int ring_next(int i) { return i + 1 == R ? 0 : i + 1; }

template <int J, int R = Ring<J>::R>
__device__ void dp_alpha_t(const Params& p, const Samp& c, int u0, int w, int nwd, int4* ring,
                           float2* xch, const int* tab) {
    constexpr int PF = R - 2;
    const int lane = threadIdx.x & 31, nthreads = nwd * 32;
    Lanes<J> L;
    lanes_init<J>(c, u0, lane, p.edge + c.off, p.alpha + c.off, L);
    float am[J];
    int ae[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        am[j] = L.u[j] == 0 ? 1.0f : 0.0f;
        ae[j] = L.u[j] == 0 ? 0 : kZeroExp;
    }
    store_diag<J>(0, 0, L, am, ae);   // alpha(0,0) = 1 (base(0) = 0)
    int4* const rl = ring + lane;
    float2* const mine = xch + w * kXch;
    const float2* const left = xch + (w > 0 ? w - 1 : 0) * kXch;
    // Step e (e = 0..D-2) forms alpha(e+1) from the records of diagonal e.
    int si = 0;
    for (int k = 0; k < PF; ++k) {
        ring_issue_t<J>(rl + si * (J * 32), k, tab[min(k, c.D - 1)], L, k < c.D);
        cp_commit();
        si = ring_next<R>(si);
    }
    const int nwork = c.D - 1;
    const int nblk = (nwork + kSkew - 1) / kSkew;
    if (nwd > 1)
        for (int k = 0; k < w; ++k) named_barrier_mem(1, nthreads);
    cp_wait_mem<PF - 1>();
    int so = 0;
    int4 edn[J];
#pragma unroll
    for (int j = 0; j < J; ++j) edn[j] = rl[j * 32];
    so = ring_next<R>(so);
    int e = 0;
    for (int bk = 0; bk < nblk; ++bk) {
#pragma unroll
        for (int k = 0; k < kSkew; ++k, ++e) {
            const bool act = e < nwork;
            int4 ed[J];
#pragma unroll
            for (int j = 0; j < J; ++j) ed[j] = edn[j];
            const int xs = (e + 1) & (kXch - 1);
            const float2 nv = left[xs];
            const int bst = tab[min(e + 1, c.D - 1)];
            {
                const int ee = e + PF;
                ring_issue_t<J>(rl + si * (J * 32), ee, tab[min(ee, c.D - 1)], L, ee < c.D);
                cp_commit();
                si = ring_next<R>(si);
            }
            cp_wait_mem<PF - 1>();
#pragma unroll
            for (int j = 0; j < J; ++j) edn[j] = rl[so * (J * 32) + j * 32];
            so = ring_next<R>(so);
            float bm[J], ym[J];
            int be[J], ye[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                xf_mul(am[j], ae[j], __int_as_float(ed[j].x), ed[j].y - kEdgeBias, bm[j], be[j]);
                xf_mul(am[j], ae[j], __int_as_float(ed[j].z), ed[j].w - kEdgeBias, ym[j], ye[j]);
            }
            if (lane == 31 && act) mine[xs] = make_float2(ym[J - 1], __int_as_float(ye[J - 1]));
            float sm[J];
            int se[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                sm[j] = __shfl_sync(0xffffffffu, ym[j], (lane + 31) & 31);
                se[j] = __shfl_sync(0xffffffffu, ye[j], (lane + 31) & 31);
            }
            const float edge_m = w > 0 ? nv.x : 0.0f;
            const int edge_e = w > 0 ? __float_as_int(nv.y) : kZeroExp;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const float nm = lane ? sm[j] : (j ? sm[j - 1] : edge_m);
                const int ne = lane ? se[j] : (j ? se[j - 1] : edge_e);
                float m;
                int x;
                if (k & 1) xf_add<true>(bm[j], be[j], nm, ne, m, x);
                else xf_add<false>(bm[j], be[j], nm, ne, m, x);
                am[j] = act ? m : am[j];
                ae[j] = act ? x : ae[j];
            }
            if (act) store_diag<J>(e + 1, bst, L, am, ae);
        }
        if (nwd > 1) named_barrier_mem(1, nthreads);
    }
    if (nwd > 1)
        for (int k = 0; k < nwd - 1 - w; ++k) named_barrier_mem(1, nthreads);
    cp_wait<0>();
    // P(y|x) = alpha(T-1,U) p_blank(T-1,U): the terminal blank (diagonal D-1).
#pragma unroll
    for (int j = 0; j < J; ++j) {
        if (L.u[j] == c.U) {
            const int4 ed = __ldcg(L.e[j] + tab[c.D - 1]);
            float m;
            int x;
            xf_mul(am[j], ae[j], __int_as_float(ed.x), ed.y - kEdgeBias, m, x);
            xf_norm(m, x);
            p.pm[c.b] = m;
            p.pe[c.b] = x;
            const double ll2 = (double)x + log2((double)m);
            p.lossa[c.b] = -ll2 * kLn2d;
            p.loss[c.b] = (float)(-ll2 * kLn2d);
        }
    }
}

template <int J, int R = Ring<J>::R>
__device__ void dp_beta_t(const Params& p, const Samp& c, int u0, int w, int nwd, int4* ring,
                          float2* xch, const int* tab) {
    constexpr int PF = R - 2;
    const int lane = threadIdx.x & 31, nthreads = nwd * 32;
    Lanes<J> L;
    lanes_init<J>(c, u0, lane, p.edge + c.off, p.beta + c.off, L);
    float vm[J];
    int ve[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        vm[j] = L.u[j] == c.U ? 1.0f : 0.0f;
        ve[j] = L.u[j] == c.U ? 0 : kZeroExp;
    }
    int4* const rl = ring + lane;
    float2* const mine = xch + w * kXch;
    const float2* const right = xch + (w + 1 < nwd ? w + 1 : w) * kXch;
    // The slot of diagonal D holds this warp's first-column start value (read
    // by warp w-1 at d = D-1, after the first barrier).
    if (lane == 0) mine[c.D & (kXch - 1)] = make_float2(vm[0], __int_as_float(ve[0]));
    // Step j (j = 0..D-1) forms beta on diagonal d = D-1-j from its records.
    int si = 0;
    for (int k = 0; k < PF; ++k) {
        const int d = c.D - 1 - k;
        ring_issue_t<J>(rl + si * (J * 32), d, tab[max(d, 0)], L, d >= 0);
        cp_commit();
        si = ring_next<R>(si);
    }
    const int nblk = (c.D + kSkew - 1) / kSkew;
    if (nwd > 1)
        for (int k = 0; k < nwd - 1 - w; ++k) named_barrier_mem(2, nthreads);
    cp_wait_mem<PF - 1>();
    int so = 0;
    int4 edn[J];
#pragma unroll
    for (int j = 0; j < J; ++j) edn[j] = rl[j * 32];
    so = ring_next<R>(so);
    int d = c.D - 1;
    for (int bk = 0; bk < nblk; ++bk) {
#pragma unroll
        for (int k = 0; k < kSkew; ++k, --d) {
            const bool act = d >= 0;
            int4 ed[J];
#pragma unroll
            for (int j = 0; j < J; ++j) ed[j] = edn[j];
            const float2 nv = right[(d + 1) & (kXch - 1)];
            const int bst = tab[max(d, 0)];
            {
                const int dd = d - PF;
                ring_issue_t<J>(rl + si * (J * 32), dd, tab[max(dd, 0)], L, dd >= 0);
                cp_commit();
                si = ring_next<R>(si);
            }
            cp_wait_mem<PF - 1>();
#pragma unroll
            for (int j = 0; j < J; ++j) edn[j] = rl[so * (J * 32) + j * 32];
            so = ring_next<R>(so);
            float sm[J];
            int se[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                sm[j] = __shfl_sync(0xffffffffu, vm[j], (lane + 1) & 31);
                se[j] = __shfl_sync(0xffffffffu, ve[j], (lane + 1) & 31);
            }
            const float edge_m = w + 1 < nwd ? nv.x : 0.0f;
            const int edge_e = w + 1 < nwd ? __float_as_int(nv.y) : kZeroExp;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const float nm = (lane < 31) ? sm[j] : (j + 1 < J ? sm[j + 1] : edge_m);
                const int ne = (lane < 31) ? se[j] : (j + 1 < J ? se[j + 1] : edge_e);
                float bm, ym, m;
                int be, ye, x;
                xf_mul(vm[j], ve[j], __int_as_float(ed[j].x), ed[j].y - kEdgeBias, bm, be);
                xf_mul(nm, ne, __int_as_float(ed[j].z), ed[j].w - kEdgeBias, ym, ye);
                if (k & 1) xf_add<true>(bm, be, ym, ye, m, x);
                else xf_add<false>(bm, be, ym, ye, m, x);
                vm[j] = act ? m : vm[j];
                ve[j] = act ? x : ve[j];
            }
            if (act) {
                store_diag<J>(d, bst, L, vm, ve);
                if (lane == 0) mine[d & (kXch - 1)] = make_float2(vm[0], __int_as_float(ve[0]));
            }
        }
        if (nwd > 1) named_barrier_mem(2, nthreads);
    }
    if (nwd > 1)
        for (int k = 0; k < w; ++k) named_barrier_mem(2, nthreads);
    cp_wait<0>();
    if (u0 == 0 && lane == 0) {
        float m = vm[0];
        int x = ve[0];
        xf_norm(m, x);
        p.lossb[c.b] = -((double)x + log2((double)m)) * kLn2d;
    }
}

// ---- One warp per direction (lattices up to 32 * kWarpDpMaxJ columns) ----
// The same recursions with a single warp per direction: lane l owns the J
// consecutive columns u = J l + j, so the label arc crosses lanes only at a
// lane's first column (alpha) or last column (beta): one shuffle pair per
// anti-diagonal, and no other warp, barrier or shared exchange.  Alone on
// their SM sub-partition the two warps issue the whole step without
// contention.  The position of diagonal d in the sample's node arrays is a
// running sum (no table, any number of diagonals): node (t, u) of diagonal d
// is at base(d) - u, base(d) = N(d) + d - max(0, d - U), and
// base(d + 1) = base(d) + min(d, T - 1) + 2 - max(0, d + 1 - U).
// Transition records of future diagonals are prefetched with zero-filling
// cp.async into a per-warp ring of R slots (slot layout [j][lane]: reads are
// bank-conflict free); small J also keeps the next diagonal's records in
// registers one step ahead.
// Measured on GB300: faster than several warps per direction for lattices of
// up to 64 columns (115 vs 146 ns per anti-diagonal on 21-41 columns), slower
// above (one warp then issues the whole step alone).
constexpr int kWarpDpMaxJ = 2;
template <int J> struct WRing {
    static constexpr int R = J <= 4 ? 16 : J <= 8 ? 8 : 4;   // ring slots (diagonals)
    static constexpr bool kRegAhead = J <= 4;                 // records one step ahead in registers
};
__host__ __device__ inline int wdp_jclass(int W) { return W <= 32 ? 1 : 2; }
__host__ __device__ inline int wdp_ring_depth(int Jc) { return Jc <= 4 ? 16 : Jc <= 8 ? 8 : 4; }
// Shared memory of the two direction warps' rings for lattices up to W columns.
__host__ __device__ inline size_t wdp_smem_bytes(int W) {
    const int Jc = wdp_jclass(W);
    return (size_t)2 * wdp_ring_depth(Jc) * Jc * 32 * sizeof(int4);
}

__device__ __forceinline__ int64_t wbase_next(int64_t b, int d, int T, int U) {
    return b + min(d, T - 1) + 2 - max(0, d + 1 - U);
}
__device__ __forceinline__ int64_t wbase_prev(int64_t b, int d, int T, int U) {
    return b - min(d - 1, T - 1) - 2 + max(0, d - U);
}
// Base of diagonal d from scratch (N(d) by inclusion-exclusion).
__device__ __forceinline__ int64_t wbase_of(int d, int T, int U) {
    return diag_start(d, T, U + 1) + d - max(0, d - U);
}

// Zero-filling copies of diagonal e's records (base be) into a ring slot:
// lane l copies the records of its columns J l .. J l + J - 1.
template <int J>
__device__ __forceinline__ void wring_issue(int4* slot, const int4* es, int64_t be, int e, int lane,
                                            int T, int U) {
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int u = J * lane + j;
        const bool ok = u <= U && (unsigned)(e - u) < (unsigned)T;
        cp16z(slot + j * 32 + lane, ok ? es + (be - u) : es, ok);
    }
}

template <int J>
__device__ __forceinline__ void wring_read(const int4* slot, int lane, int4 (&r)[J]) {
#pragma unroll
    for (int j = 0; j < J; ++j) r[j] = lds128(slot + j * 32 + lane);
}

// Forward variable on one warp: step e (e = 0..D-2) forms alpha on diagonal
// e + 1 from alpha on diagonal e and the records of diagonal e.
template <int J>
__device__ void dp_alpha_w(const Params& p, const Samp& c, int4* ring) {
    constexpr int R = WRing<J>::R, PF = R - 1;
    constexpr bool AHEAD = WRing<J>::kRegAhead;
    const int lane = threadIdx.x & 31;
    const int T = c.T, U = c.U, D = c.D;
    const int4* es = p.edge + c.off;
    int2* out = p.alpha + c.off;
    float am[J];
    int ae[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const bool origin = lane == 0 && j == 0;
        am[j] = origin ? 1.0f : 0.0f;
        ae[j] = origin ? 0 : kZeroExp;
    }
    if (lane == 0) out[0] = make_int2(__float_as_int(1.0f), 0);   // alpha(0,0) = 1
    // Prefetch diagonals 0 .. PF-1.
    int64_t bi = 0;   // base of the next diagonal to issue
    int ei = 0;
    for (; ei < PF; ++ei) {
        if (ei < D) wring_issue<J>(ring + (ei % R) * (J * 32), es, bi, ei, lane, T, U);
        cp_commit();
        bi = wbase_next(bi, ei, T, U);
    }
    int4 rc[J];
    if (AHEAD) {
        cp_wait<PF - 1>();
        wring_read<J>(ring, lane, rc);
    }
    int64_t bs = wbase_next(0, 0, T, U);   // base of diagonal e + 1 (stores)
    auto step = [&](int e, auto norm) {
        if (ei < D) wring_issue<J>(ring + (ei % R) * (J * 32), es, bi, ei, lane, T, U);
        cp_commit();
        bi = wbase_next(bi, ei, T, U);
        ++ei;
        int4 rn[J];
        // Without the register look-ahead the records are read from the ring as
        // they are used (plain loads after a memory-clobbering wait, so that
        // the compiler orders them after it but keeps few of them live).
        const int4* cur = ring + (e % R) * (J * 32) + lane;
        if (AHEAD) {
            cp_wait<PF - 1>();   // diagonal e + 1 has landed
            wring_read<J>(ring + ((e + 1) % R) * (J * 32), lane, rn);
        } else {
            cp_wait_mem<PF>();   // diagonal e has landed
        }
        auto rec = [&](int j) -> int4 { return AHEAD ? rc[j] : cur[j * 32]; };
        // Label arc into this lane's first column: the last column of lane - 1.
        float nm;
        int ne;
        {
            float ym;
            int ye;
            const int4 rl = rec(J - 1);
            xf_mul(am[J - 1], ae[J - 1], __int_as_float(rl.z), rl.w - kEdgeBias, ym, ye);
            nm = __shfl_up_sync(0xffffffffu, ym, 1);
            ne = __shfl_up_sync(0xffffffffu, ye, 1);
            if (lane == 0) {
                nm = 0.0f;
                ne = kZeroExp;
            }
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            float bm, ym;
            int be, ye;
            const int4 r = rec(j);
            xf_mul(am[j], ae[j], __int_as_float(r.x), r.y - kEdgeBias, bm, be);
            xf_mul(am[j], ae[j], __int_as_float(r.z), r.w - kEdgeBias, ym, ye);
            xf_add<decltype(norm)::value>(bm, be, nm, ne, am[j], ae[j]);
            nm = ym;
            ne = ye;
        }
        const int d = e + 1;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int u = J * lane + j;
            if (u <= U && (unsigned)(d - u) < (unsigned)T)
                out[bs - u] = make_int2(__float_as_int(am[j]), ae[j]);
        }
        bs = wbase_next(bs, d, T, U);
        if (AHEAD) {
#pragma unroll
            for (int j = 0; j < J; ++j) rc[j] = rn[j];
        }
    };
    int e = 0;
    for (; e + 1 < D - 1; e += 2) {
        step(e, std::false_type());
        step(e + 1, std::true_type());
    }
    if (e < D - 1) step(e, std::false_type());
    cp_wait<0>();
    // P(y|x) = alpha(T-1,U) p_blank(T-1,U): the terminal blank (diagonal D-1).
    const int jU = U % J;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        if (j == jU && lane == U / J) {
            const int4 ed = __ldcg(es + node_index(T - 1, U, T, U));
            float m;
            int x;
            xf_mul(am[j], ae[j], __int_as_float(ed.x), ed.y - kEdgeBias, m, x);
            xf_norm(m, x);
            p.pm[c.b] = m;
            p.pe[c.b] = x;
            const double ll2 = (double)x + log2((double)m);
            p.lossa[c.b] = -ll2 * kLn2d;
            p.loss[c.b] = (float)(-ll2 * kLn2d);
        }
    }
}

// Backward variable on one warp: step d (d = D-1..0) forms beta on diagonal d
// from beta on diagonal d + 1 (a virtual node after the terminal blank holds
// 1) and the records of diagonal d.
template <int J>
__device__ void dp_beta_w(const Params& p, const Samp& c, int4* ring) {
    constexpr int R = WRing<J>::R, PF = R - 1;
    constexpr bool AHEAD = WRing<J>::kRegAhead;
    const int lane = threadIdx.x & 31;
    const int T = c.T, U = c.U, D = c.D;
    const int4* es = p.edge + c.off;
    int2* out = p.beta + c.off;
    float vm[J];
    int ve[J];
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const bool last = J * lane + j == U;
        vm[j] = last ? 1.0f : 0.0f;
        ve[j] = last ? 0 : kZeroExp;
    }
    // Prefetch diagonals D-1 down to D-PF.
    int64_t bi = wbase_of(D - 1, T, U);   // base of the next diagonal to issue
    int di = D - 1;
    int k = 0;
    for (; k < PF; ++k, --di) {
        if (di >= 0) wring_issue<J>(ring + (k % R) * (J * 32), es, bi, di, lane, T, U);
        cp_commit();
        if (di > 0) bi = wbase_prev(bi, di, T, U);
    }
    int4 rc[J];
    if (AHEAD) {
        cp_wait<PF - 1>();
        wring_read<J>(ring, lane, rc);
    }
    int64_t bs = wbase_of(D - 1, T, U);   // base of diagonal d (stores)
    // Step number s = D-1-d uses ring slot s % R.
    auto step = [&](int s, auto norm) {
        const int d = D - 1 - s;
        if (di >= 0) wring_issue<J>(ring + ((s + PF) % R) * (J * 32), es, bi, di, lane, T, U);
        cp_commit();
        if (di > 0) bi = wbase_prev(bi, di, T, U);
        --di;
        int4 rn[J];
        const int4* cur = ring + (s % R) * (J * 32) + lane;
        if (AHEAD) {
            cp_wait<PF - 1>();   // diagonal d - 1 has landed
            wring_read<J>(ring + ((s + 1) % R) * (J * 32), lane, rn);
        } else {
            cp_wait_mem<PF>();   // diagonal d has landed (records read as used)
        }
        auto rec = [&](int j) -> int4 { return AHEAD ? rc[j] : cur[j * 32]; };
        // Label arc out of this lane's last column: the first column of lane + 1.
        float nm = __shfl_down_sync(0xffffffffu, vm[0], 1);
        int ne = __shfl_down_sync(0xffffffffu, ve[0], 1);
        if (lane == 31) {
            nm = 0.0f;
            ne = kZeroExp;
        }
#pragma unroll
        for (int j = J - 1; j >= 0; --j) {
            float bm, ym;
            int be, ye;
            const int4 r = rec(j);
            xf_mul(vm[j], ve[j], __int_as_float(r.x), r.y - kEdgeBias, bm, be);
            const float cm = vm[j];
            const int ce = ve[j];
            xf_mul(nm, ne, __int_as_float(r.z), r.w - kEdgeBias, ym, ye);
            xf_add<decltype(norm)::value>(bm, be, ym, ye, vm[j], ve[j]);
            nm = cm;
            ne = ce;
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int u = J * lane + j;
            if (u <= U && (unsigned)(d - u) < (unsigned)T)
                out[bs - u] = make_int2(__float_as_int(vm[j]), ve[j]);
        }
        if (d > 0) bs = wbase_prev(bs, d, T, U);
        if (AHEAD) {
#pragma unroll
            for (int j = 0; j < J; ++j) rc[j] = rn[j];
        }
    };
    int s = 0;
    for (; s + 1 < D; s += 2) {
        step(s, std::false_type());
        step(s + 1, std::true_type());
    }
    if (s < D) step(s, std::true_type());
    cp_wait<0>();
    if (lane == 0) {
        float m = vm[0];
        int x = ve[0];
        xf_norm(m, x);
        p.lossb[c.b] = -((double)x + log2((double)m)) * kLn2d;
    }
}

// The recursion of direction dir (0 alpha, 1 beta) on the calling warp;
// ring: that direction's ring (wdp_smem_bytes / 2).
template <int J>
__device__ __forceinline__ void dp_run_w(const Params& p, const Samp& c, int4* ring, int dir) {
    if (dir == 0) dp_alpha_w<J>(p, c, ring);
    else dp_beta_w<J>(p, c, ring);
}
__device__ __forceinline__ void dp_dispatch_w(const Params& p, const Samp& c, int4* ring, int dir) {
    if (wdp_jclass(c.W) == 1) dp_run_w<1>(p, c, ring, dir);
    else dp_run_w<2>(p, c, ring, dir);
}

// Target lattice columns per lane before another compute warp is added.
#ifndef RNNT_DP_SLOTS
#define RNNT_DP_SLOTS 1
#endif
__host__ __device__ inline int dp_warps(int W, int maxw = kDpWarps) {
    return min(maxw, (W + 32 * RNNT_DP_SLOTS - 1) / (32 * RNNT_DP_SLOTS));
}
__host__ __device__ inline int dp_slots(int W, int maxw = kDpWarps) {
    const int n = dp_warps(W, maxw);
    return (W + 32 * n - 1) / (32 * n);
}
__host__ __device__ inline int dp_jclass(int J) {
    return J <= 1 ? 1 : J <= 2 ? 2 : J <= 3 ? 3 : J <= 4 ? 4 : J <= 6 ? 6 : 8;
}
__host__ __device__ inline int dp_ring_depth(int Jc) {
    return Jc == 1 ? 16 : Jc == 2 ? 12 : Jc <= 4 ? 10 : 6;
}

// Dynamic shared memory of the DP for lattices up to W columns: the rings of
// the compute warps, then the table of diagonal bases.
__host__ __device__ inline size_t dp_ring_bytes(int W) {
    const int Jc = dp_jclass(dp_slots(W));
    return (size_t)2 * dp_warps(W) * dp_ring_depth(Jc) * Jc * 32 * sizeof(int4);
}
__host__ __device__ inline size_t dp_smem_bytes(int W) {
    return dp_ring_bytes(W) + (size_t)kTabMax * sizeof(int);
}

// The recursion of direction dir on warps w = 0 .. dp_warps(W)-1 given by the
// caller (other warps return at once); ring: the first of that direction's
// rings, xch: its exchange area, tab: the diagonal base table (filled by the
// caller when T+U <= kTabMax).
template <int J, int R = Ring<J>::R, int MAXW = kDpWarps>
__device__ __forceinline__ void dp_run_dir(const Params& p, const Samp& c, int dir, int w,
                                           int4* ring, float2* xch, const int* tab) {
    const int nwd = dp_warps(c.W, MAXW);
    if (w >= nwd) return;
    ring += (size_t)w * R * J * 32;
    if (c.D <= kTabMax) {
        if (dir == 0) dp_alpha_t<J, R>(p, c, w * 32 * J, w, nwd, ring, xch, tab);
        else dp_beta_t<J, R>(p, c, w * 32 * J, w, nwd, ring, xch, tab);
    } else {
        if (dir == 0) dp_alpha<J, R>(p, c, w * 32 * J, w, nwd, ring, xch);
        else dp_beta<J, R>(p, c, w * 32 * J, w, nwd, ring, xch);
    }
}

__device__ __forceinline__ void dp_fill_tab(const Samp& c, int* tab) {
    if (c.D <= kTabMax)
        for (int d = threadIdx.x; d < c.D; d += blockDim.x) tab[d] = diag_base(c, d);
}

// Both directions of one sample on one CTA of 8 warps (the persistent
// kernel's DP task): lattices of up to 64 columns on warps 0 (alpha) and 1
// (beta) one warp each; wider ones alpha on even and beta on odd warp ids, so
// that the two recursions run on different SM sub-partitions.  Called by
// every thread of the CTA.  xch: 2 * kDpWarps * kXch entries.
template <int J>
__device__ __forceinline__ void dp_run(const Params& p, const Samp& c, int4* smem, float2* xch) {
    const int wid = threadIdx.x >> 5;
    if (c.W <= 32 * kWarpDpMaxJ) {
        // Warps 0/1, or 2/3 in the second half of a two-CTA-per-SM grid, so
        // that two CTAs on one SM (blocks i and i + gridDim/2 in the usual
        // placement) put their four recursion warps on four sub-partitions.
        const int w = wid - ((blockIdx.x >= gridDim.x / 2) ? 2 : 0);
        if (w == 0 || w == 1)
            dp_dispatch_w(p, c, smem + (size_t)w * (wdp_smem_bytes(c.W) / 2 / sizeof(int4)), w);
        return;
    }
    int* tab = reinterpret_cast<int*>(reinterpret_cast<char*>(smem) + dp_ring_bytes(c.W));
    dp_fill_tab(c, tab);
    __syncthreads();
    const int dir = wid & 1, w = wid >> 1;
    int4* ring = smem + (size_t)dir * dp_warps(c.W) * Ring<J>::R * J * 32;
    dp_run_dir<J>(p, c, dir, w, ring, xch + dir * kDpWarps * kXch, tab);
}

// Ring depth of the per-stage recursions (one direction per CTA, up to 4
// warps): at most 96 KB of rings.
__host__ __device__ constexpr int deep_ring(int J) {
    return J <= 1 ? 24 : J <= 2 ? 16 : J <= 3 ? 12 : J <= 4 ? 10 : J <= 6 ? 8 : 6;
}
__host__ __device__ inline size_t dp_deep_ring_bytes(int W) {
    const int Jc = dp_jclass(dp_slots(W, kDpWarpsStaged));
    return (size_t)dp_warps(W, kDpWarpsStaged) * deep_ring(Jc) * Jc * 32 * sizeof(int4);
}

// Per-stage recursions: one CTA per (sample in DP order, direction =
// blockIdx.y), so that the alpha and the beta recursion of a sample run on
// different SMs (each SM's issue slots, not the recursion's dependent chain,
// bound a step when both directions share one SM).  Lattices of up to 64
// columns take one warp; wider ones dp_warps(W) warps (measured: 8 warps per
// direction are slower than 4 on a 301-column lattice, 211 vs 176 ns per
// anti-diagonal).
template <int J>
__device__ __forceinline__ void k_dp_body(const Params& p, const Samp& c, int4* smem, float2* xch) {
    const int dir = blockIdx.y;
    if (c.W <= 32 * kWarpDpMaxJ) {
        if (threadIdx.x < 32) dp_dispatch_w(p, c, smem, dir);
        return;
    }
    int* tab = reinterpret_cast<int*>(reinterpret_cast<char*>(smem) + dp_deep_ring_bytes(c.W));
    dp_fill_tab(c, tab);
    __syncthreads();
    dp_run_dir<J, deep_ring(J), kDpWarpsStaged>(p, c, dir, threadIdx.x >> 5, smem, xch, tab);
}

// Zero-fill of the gradient buffer by the CTAs of the recursion launch past
// its two per sample (blockIdx.y >= 2): every CTA zeroes its shared buffer,
// then one thread claims 1 MB chunks from a counter and writes each with bulk
// (TMA) stores of that buffer, so the fill costs the SM few instructions
// while recursions run beside it.  A CTA placed on an SM of the longest
// recursion (its CTAs record their SMs first) leaves at once.  The bytes
// past the last 16-byte boundary are stored by the thread that claims the
// last chunk.
//
// Only as many CTAs take part as keep the fill within about the longest
// recursion's duration: on GB300 a recursion step takes ~175 ns per
// anti-diagonal and one CTA's bulk stores write ~60 GB/s, ~10 KB per step.
// More CTAs saturate HBM, which slows the recursion (its transition records
// stream from HBM) without ending the call sooner (measured on a 1500 x 301
// lattice beside 830 MB of fill: 173 ns per step with 48 CTAs, 192 with 152).
constexpr int64_t kZeroChunk = 1 << 20;
constexpr int64_t kZeroBytesPerStep = 9500;
__device__ __forceinline__ void zero_fill(const Params& p, int4* smem) {
    const int z = blockIdx.x + gridDim.x * (blockIdx.y - 2);
    const int bc = __ldcg(p.order);
    const int64_t per = ((int64_t)__ldg(p.Tl + bc) + __ldg(p.Ul + bc)) * kZeroBytesPerStep;
    const int64_t need = (p.zfill + per - 1) / per;
    if (z >= min((int64_t)p.zcta, max((int64_t)8, need))) return;
    const int sm = smid();
    const volatile int32_t* ve = p.err;
    if (sm == ve[14] || sm == ve[15]) return;
    for (int i = threadIdx.x; i < p.zbuf / 16; i += blockDim.x) smem[i] = make_int4(0, 0, 0, 0);
    fence_proxy_async();   // the zeros are read by the bulk-copy (async) proxy
    __syncthreads();
    if (threadIdx.x != 0) return;
    char* g = static_cast<char*>(p.grad);
    const int64_t body = p.zfill & ~int64_t(15);
    for (;;) {
        const int64_t a = (int64_t)atomicAdd(p.err + 13, 1) * kZeroChunk;
        if (a >= p.zfill) break;
        const int64_t e = min(a + kZeroChunk, p.zfill), eb = min(e, body);
        for (int64_t x = a; x < eb; x += p.zbuf)
            tma_store(g + x, smem, (uint32_t)min((int64_t)p.zbuf, eb - x));
        tma_store_commit();
        // At most 4 further chunks' stores in flight from this CTA.
        asm volatile("cp.async.bulk.wait_group.read 4;\n" ::: "memory");
        for (int64_t x = max(a, body); x < e; ++x) g[x] = 0;
    }
    tma_store_wait_all();
}

__global__ void __launch_bounds__(32 * kDpWarpsStaged) k_dp(Params p) {
    if (*p.err) return;
    extern __shared__ int4 smem[];
    __shared__ float2 xch[kDpWarpsStaged * kXch];
    if (blockIdx.y >= 2) {
        zero_fill(p, smem);
        return;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.zfill) p.err[14 + blockIdx.y] = smid();
    Samp c;
    c.b = p.order[blockIdx.x];
    c.T = p.Tl[c.b];
    c.U = p.Ul[c.b];
    c.W = c.U + 1;
    c.D = c.T + c.U;
    c.off = p.off[c.b];
    const uint64_t t0 = (p.trace && threadIdx.x == 0) ? global_ns() : 0;
    const int J = dp_jclass(dp_slots(c.W, kDpWarpsStaged));
    if (J == 1) k_dp_body<1>(p, c, smem, xch);
    else if (J == 2) k_dp_body<2>(p, c, smem, xch);
    else if (J == 3) k_dp_body<3>(p, c, smem, xch);
    else if (J == 4) k_dp_body<4>(p, c, smem, xch);
    else if (J == 6) k_dp_body<6>(p, c, smem, xch);
    else k_dp_body<8>(p, c, smem, xch);
    if (p.trace) {   // records 2b, 2b+1 of the trace: this sample's two recursions
        __syncthreads();
        if (threadIdx.x == 0)
            trace_task(p, 2 * blockIdx.x + blockIdx.y, TASK_DP | (c.b << 2), t0);
    }
}

// ---------------------------------------------------------------- combine
// Per row: occupancy c = alpha beta / P and the arc posteriors
// alpha p_blank beta(t+1,u) / P and alpha p_label beta(t,u+1) / P, folded with
// the reduction scale into the gradient pass's per-row record
//   {log2(c scale) - lse2 (or -inf: a row of exact zeros), post_blank scale,
//    post_label scale, label id (-1 at u = U)}.
__device__ __forceinline__ float xf_to_float(float m, int e) {
    return (m == 0.0f || e < -200) ? 0.0f : ldexpf(m, min(e, 200));
}

// One row's gradient record.  Everything it reads that the same call wrote
// (alpha, beta, transition records, lse2, P) is loaded through L2 only
// (ld.global.cg): in the persistent kernel other CTAs write these while this
// SM may hold neighbouring lines in L1.
// combine_at: node (t,u) of sample b (lengths T, U; first row / node o),
// global node index i, compact row r.
__device__ __forceinline__ float4 combine_at(const Params& p, int b, int T, int U, int64_t o,
                                             int t, int u, int64_t i, int64_t r) {
    const int2 A = __ldcg(p.alpha + i), Bt = __ldcg(p.beta + i);
    const int4 Ed = __ldcg(p.edge + i);
    const float Pm = __ldcg(p.pm + b);
    const int Pe = __ldcg(p.pe + b);
    const float am = __int_as_float(A.x), bm = __int_as_float(Bt.x);
    const float inv = 1.0f / Pm;
    float lc = -INFINITY;
    if (am != 0.0f && bm != 0.0f) lc = (float)(A.y + Bt.y - Pe) + lg2(am * bm * inv);
    const int y = (u < U) ? __ldg(p.targets + (int64_t)b * p.S + u) : -1;
    // Every element of this gradient row rounds to zero (with FastEmit the
    // row's elements are bounded by (1 + fe) times the occupancy).
    if (!(lc + p.fe_l2 >= p.skip2))
        return make_float4(-INFINITY, 0.0f, 0.0f, __int_as_float(y));
    float eb = 0.0f, ey = 0.0f;
    if (t < T - 1) {
        const int2 Bn = __ldcg(p.beta + o + node_index(t + 1, u, T, U));
        const float pb = __int_as_float(Ed.x), bn = __int_as_float(Bn.x);
        if (am != 0.0f && pb != 0.0f && bn != 0.0f)
            eb = xf_to_float(am * pb * bn * inv, A.y + (Ed.y - kEdgeBias) + Bn.y - Pe);
    } else if (u == U) {
        eb = xf_to_float(am * bm * inv, A.y + Bt.y - Pe);
    }
    if (u < U) {
        const int2 Bn = __ldcg(p.beta + o + node_index(t, u + 1, T, U));
        const float py = __int_as_float(Ed.z), bn = __int_as_float(Bn.x);
        if (am != 0.0f && py != 0.0f && bn != 0.0f) {
            ey = xf_to_float(am * py * bn * inv, A.y + (Ed.w - kEdgeBias) + Bn.y - Pe);
            if (p.fe > 0.0f) {
                // FastEmit: the label term is (1 + fe) post_label, so the
                // softmax term p_k * (post_blank + (1 + fe) post_label) has
                // occupancy occ (1 + fe post_label / occ), post_label / occ =
                // p_label beta(t,u+1) / beta(t,u).
                const float ratio = xf_to_float(py * bn / bm, (Ed.w - kEdgeBias) + Bn.y - Bt.y);
                lc += lg2(fmaf(p.fe, ratio, 1.0f));
                ey *= 1.0f + p.fe;
            }
        }
    }
    // (Without the log-softmax lse2 is 0 for every row.)
    return make_float4(lc + p.lscale - (p.fused ? __ldcg(p.lse2 + r) : 0.0f), eb * p.scale,
                       ey * p.scale, __int_as_float(y));
}
__device__ __forceinline__ float4 combine_row(const Params& p, int64_t r, int b) {
    const int T = __ldg(p.Tl + b), U = __ldg(p.Ul + b), W = U + 1;
    const int64_t o = __ldcg(p.off + b);
    const unsigned rr = (unsigned)(r - o);
    const int t = (int)(rr / (unsigned)W), u = (int)(rr - (unsigned)t * W);
    return combine_at(p, b, T, U, o, t, u, o + node_index(t, u, T, U), r);
}

// Long rows: every row's gradient record, ahead of the gradient kernel.
__global__ void __launch_bounds__(256) k_combine(Params p) {
    if (*p.err) return;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int b = (r < nodes(p)) ? find_sample(p.off, p.B, r) : 0;
    for (; r < nodes(p); r += stride) {
        b = advance_sample(p.off, p.B, b, r);
        p.info[r] = combine_row(p, r, b);
    }
}

// The gradient record of row r for a lane that walks increasing rows (b: the
// lane's current sample, -1 before its first row); a zero-row record for
// lanes without a row.
__device__ __forceinline__ float4 row_record(const Params& p, int64_t r, bool valid, int& b) {
    if (!valid) return make_float4(-INFINITY, 0.0f, 0.0f, __int_as_float(-1));
    b = b < 0 ? find_sample(p.off, p.B, r) : advance_sample(p.off, p.B, b, r);
    return combine_row(p, r, b);
}

__device__ void finalize_block(const Params& p);

// End of the last kernel of a per-stage call: every CTA publishes its writes
// and counts itself out; the last one runs the loss check and reduction
// (finalize_block, 256 threads), so no separate launch is needed.
__device__ __forceinline__ void finalize_if_last(const Params& p) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&p.err[8], 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (s_last) {
        __threadfence();
        finalize_block(p);
    }
}

// ---------------------------------------------------------------- grad pass
// grad_k * scale = 2^(h_k log2 e + log2(c scale) - lse2) - [k=blank] post_blank
// scale - [k=y] post_label scale, clipped to +-clamp*scale (clip-then-scale).
// Long rows (kLongRowBytes and more), a whole warp per row: rows
// grid-strided over the warps so that the warps stream neighbouring rows;
// each row's record comes from the record pass (k_combine), the next one's
// loaded while the current row streams.  Few registers (the whole SM's
// threads stream); k_finalize runs the loss check after it.
template <typename Tin, bool VEC, bool FUSED>
__global__ void __launch_bounds__(256) k_grad_long(Params p) {
    if (*p.err) return;
    using E = Elt<Tin>;
    constexpr int EPV = E::kPerVec, G = 32;
    const Tin* X = static_cast<const Tin*>(p.logits);
    Tin* Y = static_cast<Tin*>(p.grad);
    const int V = p.V;
    const int lane = threadIdx.x & 31;
    const float cl = p.clamp * p.scale;
    const bool clip = p.clamp < INFINITY;
    const int vb = p.blank / EPV, eb_i = p.blank % EPV;
    const int64_t nr = nodes(p);
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
    float4 rec_next = gw < nr ? __ldcg(p.info + gw) : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t r = gw; r < nr; r += nwarps) {
        const float4 rec = rec_next;
        if (r + nwarps < nr) rec_next = __ldcg(p.info + r + nwarps);
        const float w2 = rec.x, eb = rec.y, ey = rec.z;
        const int y = __float_as_int(rec.w);
        const int64_t lr = lrow(p, r);
        const bool zero = w2 == -INFINITY;
        const Tin* row = X + lr * (int64_t)V;
        Tin* out = Y + lr * (int64_t)V;
        if (VEC) {
            const int nvec = V / EPV;
            const int vy = y >= 0 ? y / EPV : -1, ey_i = y >= 0 ? y % EPV : 0;
            const uint4* rv = reinterpret_cast<const uint4*>(row);
            uint4* ov = reinterpret_cast<uint4*>(out);
            for (int vi = lane; vi < nvec; vi += G) {
                float g[EPV];
                if (FUSED && !zero) {
                    float x[EPV];
                    E::unpack(__ldcs(rv + vi), x);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) g[e] = ex2(fmaf(x[e], kLog2e, w2));
                } else {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) g[e] = 0.0f;
                }
                if (vi == vb) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (e == eb_i) g[e] -= eb;
                }
                if (vi == vy) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (e == ey_i) g[e] -= ey;
                }
                if (clip) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) g[e] = fminf(fmaxf(g[e], -cl), cl);
                }
                __stcs(ov + vi, E::pack(g));
            }
        } else {
            for (int k = lane; k < V; k += G) {
                float gv = (FUSED && !zero) ? ex2(fmaf(E::to_f(row[k]), kLog2e, w2)) : 0.0f;
                if (k == p.blank) gv -= eb;
                if (k == y) gv -= ey;
                if (clip) gv = fminf(fmaxf(gv, -cl), cl);
                out[k] = E::from_f(gv);
            }
        }
    }
}

// Each warp takes batches of 32 consecutive rows: every lane forms one row's
// record (occupancy, arc posteriors: combine_row), then groups of G lanes write
// the rows, taking each row's record from its lane by shuffle.  The last CTA
// finishes the call (loss check, reduction).
template <typename Tin, int G, bool VEC, bool FUSED>
__global__ void __launch_bounds__(256) k_grad(Params p) {
    if (*p.err == 0) {
        using E = Elt<Tin>;
        constexpr int EPV = E::kPerVec, NG = 32 / G;
        constexpr unsigned F = 0xffffffffu;
        const Tin* X = static_cast<const Tin*>(p.logits);
        Tin* Y = static_cast<Tin*>(p.grad);
        const int V = p.V;
        const int wl = threadIdx.x & 31, lane = wl & (G - 1), grp = wl / G;
        const float cl = p.clamp * p.scale;
        const bool clip = p.clamp < INFINITY;
        const int vb = p.blank / EPV, eb_i = p.blank % EPV;
        const int64_t nr = nodes(p), nbatch = (nr + 31) / 32;
        const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
        const bool flat = flat_rows(V, sizeof(Tin), p.fused) && !p.padded;
        int bs = -1;   // this lane's sample
        // The records of a batch are formed one batch ahead of its rows.
        auto batch_rec = [&](int64_t bt, int64_t& lr) -> float4 {
            const int64_t r = bt * 32 + wl;
            const bool valid = bt < nbatch && r < nr;
            const float4 rec = row_record(p, r, valid, bs);
            lr = !valid ? 0 : p.padded ? lrow_s(p, r, bs, __ldcg(p.off + bs), __ldg(p.Ul + bs) + 1) : r;
            return rec;
        };
        int64_t bt = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
        int64_t lr_next = 0;
        float4 rec_next = batch_rec(bt, lr_next);
        for (; bt < nbatch; bt += nwarps) {
            const int64_t r0 = bt * 32;
            const int n = (int)min((int64_t)32, nr - r0);
            const float4 rec = rec_next;
            const int64_t lr_mine = lr_next;
            rec_next = batch_rec(bt + nwarps, lr_next);
            if (!VEC && FUSED && flat) {   // short rows: flat element order
                flat_grad<Tin>(p, r0, n, wl, [&](int i) {
                    return make_float4(__shfl_sync(F, rec.x, i), __shfl_sync(F, rec.y, i),
                                       __shfl_sync(F, rec.z, i), __shfl_sync(F, rec.w, i));
                });
                continue;
            }
            for (int it = 0; it * NG < n; ++it) {
                const int ri = it * NG + grp;
                const float w2 = __shfl_sync(F, rec.x, ri), eb = __shfl_sync(F, rec.y, ri);
                const float ey = __shfl_sync(F, rec.z, ri);
                const int y = __shfl_sync(F, __float_as_int(rec.w), ri);
                const int64_t lr = __shfl_sync(F, lr_mine, ri);
                if (ri >= n) continue;
                const bool zero = w2 == -INFINITY;
                const Tin* row = X + lr * (int64_t)V;
                Tin* out = Y + lr * (int64_t)V;
                if (VEC) {
                    const int nvec = V / EPV;
                    const int vy = y >= 0 ? y / EPV : -1, ey_i = y >= 0 ? y % EPV : 0;
                    const uint4* rv = reinterpret_cast<const uint4*>(row);
                    uint4* ov = reinterpret_cast<uint4*>(out);
                    for (int vi = lane; vi < nvec; vi += G) {
                        float g[EPV];
                        if (FUSED && !zero) {
                            float x[EPV];
                            E::unpack(__ldcs(rv + vi), x);
#pragma unroll
                            for (int e = 0; e < EPV; ++e) g[e] = ex2(fmaf(x[e], kLog2e, w2));
                        } else {
#pragma unroll
                            for (int e = 0; e < EPV; ++e) g[e] = 0.0f;
                        }
                        if (vi == vb) {
#pragma unroll
                            for (int e = 0; e < EPV; ++e)
                                if (e == eb_i) g[e] -= eb;
                        }
                        if (vi == vy) {
#pragma unroll
                            for (int e = 0; e < EPV; ++e)
                                if (e == ey_i) g[e] -= ey;
                        }
                        if (clip) {
#pragma unroll
                            for (int e = 0; e < EPV; ++e) g[e] = fminf(fmaxf(g[e], -cl), cl);
                        }
                        __stcs(ov + vi, E::pack(g));
                    }
                } else {
                    // Rows that are not 16-byte vectors: elements k = lane + G q, the
                    // loads of eight of them issued together.
                    constexpr int KQ = 8;
                    for (int k0 = lane; k0 < V; k0 += G * KQ) {
                        float x[KQ];
#pragma unroll
                        for (int q = 0; q < KQ; ++q) {
                            const int k = k0 + G * q;
                            x[q] = (FUSED && !zero && k < V) ? E::to_f(row[k]) : 0.0f;
                        }
#pragma unroll
                        for (int q = 0; q < KQ; ++q) {
                            const int k = k0 + G * q;
                            if (k >= V) break;
                            float gv = (FUSED && !zero) ? ex2(fmaf(x[q], kLog2e, w2)) : 0.0f;
                            if (k == p.blank) gv -= eb;
                            if (k == y) gv -= ey;
                            if (clip) gv = fminf(fmaxf(gv, -cl), cl);
                            out[k] = E::from_f(gv);
                        }
                    }
                }
            }
        }
    }
    finalize_if_last(p);
}

// Anti-diagonal of node k (0 <= k < T W) of a T x W lattice in the
// anti-diagonal-packed order: a first guess from the lattice's three parts
// (diagonal lengths rising 1 .. m-1, then m, then falling; m = min(T, W)),
// corrected against diag_start.
__device__ __forceinline__ int node_diag(int64_t k, int T, int W) {
    const int m = min(T, W), M = max(T, W), D = T + W - 1;
    const int64_t head = (int64_t)(m - 1) * m / 2;
    int d;
    if (k < head) {
        d = (int)((sqrtf(8.0f * (float)k + 1.0f) - 1.0f) * 0.5f);
    } else if (k < head + (int64_t)(M - m + 1) * m) {
        d = m - 1 + (int)((k - head) / m);
    } else {
        const int64_t kr = (int64_t)T * W - 1 - k;
        d = D - 1 - (int)((sqrtf(8.0f * (float)kr + 1.0f) - 1.0f) * 0.5f);
    }
    d = max(0, min(d, D - 1));
    while (d > 0 && diag_start(d, T, W) > k) --d;
    while (d + 1 < D && diag_start(d + 1, T, W) <= k) ++d;
    return d;
}

template <typename Tin>
__device__ __forceinline__ uint32_t elt_bits(Tin v) {
    if constexpr (sizeof(Tin) == 4) {
        uint32_t x;
        memcpy(&x, &v, 4);
        return x;
    } else {
        uint16_t x;
        memcpy(&x, &v, 2);
        return x;
    }
}

// Stores elements k1 (bits v1, if w1) and k2 (bits v2, if w2) of a gradient
// row whose other elements are already zero.  The aligned 32-byte sector
// holding an element, when it lies inside the row, is written whole (zeros
// around the value, both elements when they share it), so that no partial
// sector is left for the memory system to merge; otherwise the element alone.
template <typename Tin>
__device__ __forceinline__ void put_sparse(Tin* row, int V, int k1, uint32_t v1, bool w1, int k2,
                                           uint32_t v2, bool w2) {
    constexpr int S = sizeof(Tin);
    const uintptr_t base = reinterpret_cast<uintptr_t>(row), end = base + (uintptr_t)V * S;
    const uintptr_t e1 = base + (uintptr_t)k1 * S, e2 = base + (uintptr_t)k2 * S;
    const uintptr_t a1 = e1 & ~uintptr_t(31), a2 = e2 & ~uintptr_t(31);
    const bool in1 = a1 >= base && a1 + 32 <= end, in2 = a2 >= base && a2 + 32 <= end;
    // The sector at a with the value bits x1 at byte offset o1 and x2 at o2
    // (an offset of -1: none).
    auto sector = [](uintptr_t a, int o1, uint32_t x1, int o2, uint32_t x2) {
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t v = 0;
            if (o1 >= 0 && (o1 >> 2) == j) v |= S == 4 ? x1 : x1 << ((o1 & 2) * 8);
            if (o2 >= 0 && (o2 >> 2) == j) v |= S == 4 ? x2 : x2 << ((o2 & 2) * 8);
            w[j] = v;
        }
        uint4* q = reinterpret_cast<uint4*>(a);
        q[0] = make_uint4(w[0], w[1], w[2], w[3]);
        q[1] = make_uint4(w[4], w[5], w[6], w[7]);
    };
    auto single = [](uintptr_t e, uint32_t v) {
        if constexpr (S == 4) *reinterpret_cast<uint32_t*>(e) = v;
        else *reinterpret_cast<uint16_t*>(e) = (uint16_t)v;
    };
    if (w1 && w2 && in1 && a1 == a2) {
        sector(a1, (int)(e1 - a1), v1, (int)(e2 - a1), v2);
        return;
    }
    if (w1) {
        if (in1) sector(a1, (int)(e1 - a1), v1, -1, 0u);
        else single(e1, v1);
    }
    if (w2) {
        if (in2) sector(a2, (int)(e2 - a2), v2, -1, 0u);
        else single(e2, v2);
    }
}

// Calls without the in-kernel log-softmax, the gradient buffer already
// zeroed by the recursion launch: a row's only non-zero elements are at the
// blank and the label, -post_blank and -post_label times the reduction scale,
// clipped.  A CTA takes 1024 consecutive lattice nodes in the anti-diagonal
// order of the node arrays (so that their reads coalesce), four per thread
// with their loads issued together, the samples of its first and last node
// looked up once.  An element is stored only where its value is not exactly
// zero, so the buffer ends bit for bit as the full-row pass leaves it.  The
// last CTA runs the loss check.
constexpr int kSparseRows = 1024;
template <typename Tin>
__global__ void __launch_bounds__(256) k_grad_sparse(Params p) {
    const int64_t nr = nodes(p);
    const int64_t n0 = (int64_t)blockIdx.x * kSparseRows;
    if (*p.err == 0 && n0 < nr) {
        using E = Elt<Tin>;
        constexpr int NR = kSparseRows / 256;
        __shared__ int s_lo, s_hi;
        if (threadIdx.x < 32) {
            const int v = find_sample_warp(p.off, p.B, n0);
            if (threadIdx.x == 0) s_lo = v;
        } else if (threadIdx.x < 64) {
            const int v = find_sample_warp(p.off, p.B, min(n0 + kSparseRows - 1, nr - 1));
            if (threadIdx.x == 32) s_hi = v;
        }
        __syncthreads();
        Tin* Y = static_cast<Tin*>(p.grad);
        const float cl = p.clamp * p.scale;
        const bool clip = p.clamp < INFINITY;
        float4 rec[NR];
        int64_t lr[NR];
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            const int64_t i = n0 + threadIdx.x + 256 * k;
            rec[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            lr[k] = 0;
            if (i < nr) {
                int lo = s_lo, hi = s_hi + 1;
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (__ldcg(p.off + mid) <= i) lo = mid; else hi = mid;
                }
                const int T = __ldg(p.Tl + lo), U = __ldg(p.Ul + lo), W = U + 1;
                const int64_t o = __ldcg(p.off + lo), kk = i - o;
                const int d = node_diag(kk, T, W);
                const int t = (int)(kk - diag_start(d, T, W)) + max(0, d - U), u = d - t;
                const int64_t r = o + (int64_t)t * W + u;
                rec[k] = combine_at(p, lo, T, U, o, t, u, i, r);
                lr[k] = p.padded ? ((int64_t)lo * p.maxT + t) * p.maxW + u : r;
            }
        }
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            float gb = 0.0f - rec[k].y, gy = 0.0f - rec[k].z;
            if (clip) {
                gb = fminf(fmaxf(gb, -cl), cl);
                gy = fminf(fmaxf(gy, -cl), cl);
            }
            const int y = __float_as_int(rec[k].w);
            put_sparse<Tin>(Y + lr[k] * (int64_t)p.V, p.V, p.blank, elt_bits(E::from_f(gb)),
                            rec[k].y != 0.0f, y < 0 ? 0 : y, elt_bits(E::from_f(gy)),
                            rec[k].z != 0.0f);
        }
    }
    finalize_if_last(p);
}

// Row pass without the log-softmax: each node's two transition
// probabilities (and every big blank's) read straight from its row's
// log-probabilities, the nodes taken in the anti-diagonal order of the node
// arrays so that the records' stores coalesce: a CTA takes 1024 consecutive
// nodes, four per thread with their loads issued together, the samples of its
// first and last node looked up once.  (lse2, 0 for every such row, is never
// read, so it is not stored.)
constexpr int kGatherNodes = 1024;
template <typename Tin>
__global__ void __launch_bounds__(256) k_row_gather(Params p) {
    const int64_t nr = nodes(p);
    const int64_t n0 = (int64_t)blockIdx.x * kGatherNodes;
    if (*p.err || n0 >= nr) return;
    using E = Elt<Tin>;
    constexpr int NR = kGatherNodes / 256;
    __shared__ int s_lo, s_hi;
    if (threadIdx.x < 32) {
        const int v = find_sample_warp(p.off, p.B, n0);
        if (threadIdx.x == 0) s_lo = v;
    } else if (threadIdx.x < 64) {
        const int v = find_sample_warp(p.off, p.B, min(n0 + kGatherNodes - 1, nr - 1));
        if (threadIdx.x == 32) s_hi = v;
    }
    __syncthreads();
    const Tin* X = static_cast<const Tin*>(p.logits);
    const Tin* row[NR];
    float hb[NR], hy[NR];
    int tt[NR], uu[NR], TT[NR], UU[NR];
#pragma unroll
    for (int k = 0; k < NR; ++k) {
        const int64_t i = n0 + threadIdx.x + 256 * k;
        row[k] = nullptr;
        hb[k] = hy[k] = 0.0f;
        tt[k] = uu[k] = TT[k] = UU[k] = 0;
        if (i < nr) {
            int lo = s_lo, hi = s_hi + 1;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (__ldcg(p.off + mid) <= i) lo = mid; else hi = mid;
            }
            const int T = __ldg(p.Tl + lo), U = __ldg(p.Ul + lo), W = U + 1;
            const int64_t o = __ldcg(p.off + lo), kk = i - o;
            const int d = node_diag(kk, T, W);
            const int t = (int)(kk - diag_start(d, T, W)) + max(0, d - U), u = d - t;
            const int64_t lr = p.padded ? ((int64_t)lo * p.maxT + t) * p.maxW + u
                                        : o + (int64_t)t * W + u;
            row[k] = X + lr * (int64_t)p.V;
            hb[k] = E::get(row[k], p.blank);
            if (u < U) hy[k] = E::get(row[k], __ldg(p.targets + (int64_t)lo * p.S + u));
            tt[k] = t;
            uu[k] = u;
            TT[k] = T;
            UU[k] = U;
        }
    }
#pragma unroll
    for (int k = 0; k < NR; ++k) {
        if (!row[k]) continue;
        const int64_t i = n0 + threadIdx.x + 256 * k;
        const int t = tt[k], u = uu[k], T = TT[k], U = UU[k];
        if (!(hb[k] < INFINITY) || !(hy[k] < INFINITY)) atomicOr(p.err, ERR_NONFINITE);
        float bm = 0.0f, ym = 0.0f;
        int be = kZeroExp, ye = kZeroExp;
        if (!(t == T - 1 && u < U)) xf_prob(hb[k], 0.0f, 1.0f, bm, be);
        if (u < U) xf_prob(hy[k], 0.0f, 1.0f, ym, ye);
        p.edge[i] = make_int4(__float_as_int(bm), be + kEdgeBias, __float_as_int(ym), ye + kEdgeBias);
        for (int j = 0; j < p.K; ++j) {   // multi-blank: every big blank's probability
            float m;
            int e;
            xf_prob(E::get(row[k], p.bb_id[j]), 0.0f, 1.0f, m, e);
            p.pbb[(int64_t)j * p.rows + i] = make_int2(__float_as_int(m), e + kEdgeBias);
        }
    }
}

// Gradient rows of the multi-blank loss.  A warp takes 32 consecutive rows:
// each lane first forms one row's record (occupancy and every arc's
// posterior, all its loads issued together), then the warp writes the rows
// one by one, p_k * occ (fused) minus the posteriors at their outputs,
// clipped and scaled; FastEmit scales the label arc.  Rows whose every
// element rounds to zero are written without reading the logits.
struct MbRec {
    float w2, eb, ey;
    int y;
    int64_t lr;   // logits / gradient row
    bool zero;
    float ebb[RNNT_MAX_BIG_BLANKS];
};

__device__ __forceinline__ MbRec mb_record(const Params& p, int64_t r, int b) {
    MbRec q;
    const float c = p.bb_c;
    const int T = __ldg(p.Tl + b), U = __ldg(p.Ul + b), W = U + 1;
    const int64_t o = __ldcg(p.off + b);
    const unsigned rr = (unsigned)(r - o);
    const int t = (int)(rr / (unsigned)W), u = (int)(rr - (unsigned)t * W);
    const int64_t nd = o + node_index(t, u, T, U);
    // Inside the band of full-length anti-diagonals (U <= t + u, the node k
    // frames later still before frame T - u), node (t + k, u) is k W nodes
    // further and (t, u + 1) W - 1 further.
    const int d = t + u;
    auto down = [&](int k) { return (d >= U && d + k <= T - 1) ? nd + (int64_t)k * W
                                                                : o + node_index(t + k, u, T, U); };
    const int2 A = __ldcg(p.alpha + nd), Bt = __ldcg(p.beta + nd);
    const int4 Ed = __ldcg(p.edge + nd);
    const int2 Bb = (t + 1 < T) ? __ldcg(p.beta + down(1)) : make_int2(0, 0);
    const int2 By = (u < U) ? __ldcg(p.beta + ((d >= U && d + 1 <= T - 1)
                                                   ? nd + W - 1
                                                   : o + node_index(t, u + 1, T, U)))
                            : make_int2(0, 0);
    int2 Qb[RNNT_MAX_BIG_BLANKS], Bq[RNNT_MAX_BIG_BLANKS];
#pragma unroll
    for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) {
        Qb[i] = make_int2(0, 0);
        Bq[i] = make_int2(0, 0);
        if (i < p.K) {
            const int t1 = t + p.bb_dur[i];
            Qb[i] = __ldcg(p.pbb + (int64_t)i * p.rows + nd);
            if (t1 < T) Bq[i] = __ldcg(p.beta + down(p.bb_dur[i]));
        }
    }
    const float Pm = __ldcg(p.pm + b);
    const int Pe = __ldcg(p.pe + b);
    const float am = __int_as_float(A.x), bm = __int_as_float(Bt.x), inv = 1.0f / Pm;
    q.y = (u < U) ? __ldg(p.targets + (int64_t)b * p.S + u) : -1;
    float lc = -INFINITY;
    if (am != 0.0f && bm != 0.0f) lc = (float)(A.y + Bt.y - Pe) + lg2(am * bm * inv);
    // posterior of an arc with probability (qm, qe) into a node of beta (nm, ne)
    auto post = [&](float qm, int qe, float nm, int ne) -> float {
        if (am == 0.0f || qm == 0.0f || nm == 0.0f) return 0.0f;
        return xf_to_float(am * qm * c * nm * inv, A.y + qe + ne - Pe);
    };
    q.eb = 0.0f;
    q.ey = 0.0f;
    if (t + 1 < T) q.eb = post(__int_as_float(Ed.x), Ed.y - kEdgeBias, __int_as_float(Bb.x), Bb.y);
    else if (u == U) q.eb = post(__int_as_float(Ed.x), Ed.y - kEdgeBias, 1.0f, 0);
    if (u < U) {
        q.ey = post(__int_as_float(Ed.z), Ed.w - kEdgeBias, __int_as_float(By.x), By.y);
        if (p.fe > 0.0f && q.ey != 0.0f && bm != 0.0f) {
            // FastEmit: occupancy occ (1 + fe post_label / occ)
            const float ratio = xf_to_float(__int_as_float(Ed.z) * c * __int_as_float(By.x) / bm,
                                            (Ed.w - kEdgeBias) + By.y - Bt.y);
            lc += lg2(fmaf(p.fe, ratio, 1.0f));
            q.ey *= 1.0f + p.fe;
        }
    }
#pragma unroll
    for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) {
        q.ebb[i] = 0.0f;
        if (i >= p.K) continue;
        const int t1 = t + p.bb_dur[i];
        const float qm = __int_as_float(Qb[i].x);
        const int qe = Qb[i].y - kEdgeBias;
        if (t1 == T && u == U) q.ebb[i] = post(qm, qe, 1.0f, 0);
        else if (t1 < T) q.ebb[i] = post(qm, qe, __int_as_float(Bq[i].x), Bq[i].y);
    }
    q.zero = !(lc + p.fe_l2 >= p.skip2);
    q.w2 = q.zero ? -INFINITY : lc + p.lscale - (p.fused ? __ldcg(p.lse2 + r) : 0.0f);
    q.lr = lrow_s(p, r, b, o, W);
    return q;
}

// Gradient pass with TMA staging (16-byte aligned rows of <= 32*NV vectors).
// Each warp walks its 32-row batches; the per-row records of a batch are
// loaded one per lane (the next batch's one batch ahead), rows of exact zeros
// are stored without reading the logits, and only the remaining rows are
// fetched into the warp's stage ring, up to kStages rows ahead.  MB: the
// multi-blank loss (records from mb_record, and every big blank's arc
// posterior subtracted at its output; the vectors holding a big-blank output
// are known per lane up front, so the common vector pays one bit test).
template <typename Tin, int NV, bool MB = false>
__global__ void __launch_bounds__(256) k_grad_tma(Params p) {
    if (*p.err) {
        finalize_if_last(p);
        return;
    }
    using E = Elt<Tin>;
    constexpr int EPV = E::kPerVec;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int nw = blockDim.x >> 5, wid = threadIdx.x >> 5, wl = threadIdx.x & 31;
    const int sb = p.stage_bytes;
    unsigned char* buf = smem_raw + (size_t)wid * kStages * sb;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (size_t)nw * kStages * sb) + wid * kStages;
    if (wl == 0) {
#pragma unroll
        for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const Tin* X = static_cast<const Tin*>(p.logits);
    Tin* Y = static_cast<Tin*>(p.grad);
    const int V = p.V, nvec = V / EPV;
    const uint32_t rb = (uint32_t)V * sizeof(Tin);
    const float cl = p.clamp * p.scale;
    const bool clip = p.clamp < INFINITY;
    const int vb = p.blank / EPV, eb_i = p.blank % EPV;
    WarpRows seq;
    seq.init(nodes(p), (int64_t)blockIdx.x * nw + wid, (int64_t)gridDim.x * nw);
    const int64_t nb = (seq.count + 31) / 32;   // batches of this warp

    int bs = -1;   // this lane's sample (its rows increase along the sequence)
    // MB: per lane, the vectors (bit v: vector wl + 32 v) holding a big blank's output.
    uint32_t bbmask = 0;
    if (MB)
        for (int i = 0; i < p.K; ++i) {
            const int vi = p.bb_id[i] / EPV;
            if ((vi & 31) == wl) bbmask |= 1u << (vi >> 5);
        }
    float ebb_cur[RNNT_MAX_BIG_BLANKS], ebb_nxt[RNNT_MAX_BIG_BLANKS];
    auto load_info = [&](int64_t j, float (&ebb)[RNNT_MAX_BIG_BLANKS]) -> float4 {
        const int64_t k = j * 32 + wl;
        const bool valid = j < nb && k < seq.count;
        if (!MB) return row_record(p, valid ? seq.row(k) : 0, valid, bs);
#pragma unroll
        for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) ebb[i] = 0.0f;
        if (!valid) return make_float4(-INFINITY, 0.f, 0.f, __int_as_float(-1));
        const int64_t r = seq.row(k);
        bs = bs < 0 ? find_sample(p.off, p.B, r) : advance_sample(p.off, p.B, bs, r);
        const MbRec q = mb_record(p, r, bs);
        const float sc = q.zero ? 0.0f : p.scale;   // a zero row stays exactly zero
#pragma unroll
        for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) ebb[i] = q.ebb[i] * sc;
        return make_float4(q.w2, q.eb * sc, q.ey * sc, __int_as_float(q.y));
    };
    float4 cur = load_info(0, ebb_cur), nxt = load_info(1, ebb_nxt);
    // Rows still to be fetched, as bit masks over the current and the next batch.
    uint32_t pend_cur = __ballot_sync(0xffffffffu, cur.x != -INFINITY);
    uint32_t pend_nxt = 0;
    bool nxt_known = false;
    int64_t issued = 0, consumed = 0;
    int64_t j = 0;   // current batch

    auto issue_more = [&]() {
        while (issued - consumed < kStages) {
            if (!pend_cur && !nxt_known && j + 1 < nb) {
                pend_nxt = __ballot_sync(0xffffffffu, nxt.x != -INFINITY);
                nxt_known = true;
            }
            int64_t row;
            if (pend_cur) {
                const int bit = __ffs(pend_cur) - 1;
                pend_cur &= pend_cur - 1;
                row = seq.row(j * 32 + bit);
            } else if (nxt_known && pend_nxt) {
                const int bit = __ffs(pend_nxt) - 1;
                pend_nxt &= pend_nxt - 1;
                row = seq.row((j + 1) * 32 + bit);
            } else {
                break;
            }
            const int st = (int)(issued % kStages);
            if (wl == 0) {
                fence_proxy_async();
                tma_row_load(buf + st * sb, X + lrow(p, row) * (int64_t)V, rb, &bars[st]);
            }
            ++issued;
        }
    };

    issue_more();
    bool ok = true;
    for (; j < nb && ok; ++j) {
        const int nrows = (int)min((int64_t)32, seq.count - j * 32);
        for (int it = 0; it < nrows; ++it) {
            const int64_t r = seq.row(j * 32 + it);
            const float w2 = __shfl_sync(0xffffffffu, cur.x, it);
            const float eb = __shfl_sync(0xffffffffu, cur.y, it);
            const float ey = __shfl_sync(0xffffffffu, cur.z, it);
            const int y = __shfl_sync(0xffffffffu, __float_as_int(cur.w), it);
            const int vy = y >= 0 ? y / EPV : -1, ey_i = y >= 0 ? y % EPV : 0;
            float ebb[RNNT_MAX_BIG_BLANKS];
            if (MB) {
#pragma unroll
                for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i)
                    ebb[i] = i < p.K ? __shfl_sync(0xffffffffu, ebb_cur[i], it) : 0.0f;
            }
            uint4* ov = reinterpret_cast<uint4*>(Y + lrow(p, r) * (int64_t)V);
            const bool zero = w2 == -INFINITY;
            const uint4* rv = nullptr;
            int st = 0;
            if (!zero) {
                st = (int)(consumed % kStages);
                if (!mbar_wait(&bars[st], (uint32_t)((consumed / kStages) & 1), p.err)) {
                    ok = false;
                    break;
                }
                rv = reinterpret_cast<const uint4*>(buf + st * sb);
            }
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                const int vi = wl + 32 * i;
                if (vi >= nvec) continue;
                float g[EPV];
                if (!zero) {
                    float x[EPV];
                    E::unpack(rv[vi], x);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) g[e] = ex2(fmaf(x[e], kLog2e, w2));
                } else {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) g[e] = 0.0f;
                }
                if (vi == vb) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (e == eb_i) g[e] -= eb;
                }
                if (vi == vy) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        if (e == ey_i) g[e] -= ey;
                }
                if (MB && ((bbmask >> i) & 1u) && !zero) {
#pragma unroll
                    for (int q = 0; q < RNNT_MAX_BIG_BLANKS; ++q) {
                        if (q >= p.K) break;
                        const int k = p.bb_id[q] - vi * EPV;
#pragma unroll
                        for (int e = 0; e < EPV; ++e)
                            if (e == k) g[e] -= ebb[q];
                    }
                }
                if (clip) {
#pragma unroll
                    for (int e = 0; e < EPV; ++e) g[e] = fminf(fmaxf(g[e], -cl), cl);
                }
                __stcs(ov + vi, E::pack(g));
            }
            if (!zero) {
                __syncwarp();
                ++consumed;
                issue_more();
            }
        }
        // Advance to the next batch: its record is already loaded; fetch the one after.
        cur = nxt;
        if (MB) {
#pragma unroll
            for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) ebb_cur[i] = ebb_nxt[i];
        }
        if (!nxt_known) pend_nxt = __ballot_sync(0xffffffffu, cur.x != -INFINITY);
        pend_cur = pend_nxt;
        pend_nxt = 0;
        nxt_known = false;
        nxt = load_info(j + 2, ebb_nxt);
        if (j + 1 < nb) {
            ++j;
            issue_more();
            --j;
        }
    }
    // Drain copies still in flight (only after a timeout) before the CTA exits.
    if (!ok)
        for (int64_t k = consumed; k < issued; ++k)
            mbar_wait(&bars[k % kStages], (uint32_t)((k / kStages) & 1), p.err);
    finalize_if_last(p);
}

// ---------------------------------------------------------------- persistent kernel
// One cooperative launch runs every row, DP and gradient task of the call.
// A CTA takes the next task index from a global counter; the queue order
// (built by k_prepare) puts each sample's row chunks before its DP task and
// every DP task before the gradient chunks, so a task only ever waits on
// tasks that were handed out earlier to CTAs that are running (all CTAs are
// co-resident under a cooperative launch).  The DP of a sample therefore runs
// on one CTA while the others stream the rows of later samples and the
// gradients of earlier ones.  Waits are bounded; a timeout raises an error
// flag, releases the waiters downstream and makes every CTA stop.
constexpr int kSpinLimit = 1 << 24;

__device__ __forceinline__ int ld_acquire(const int32_t* a) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];\n" : "=r"(v) : "l"(a) : "memory");
    return v;
}
// Warp: rows [r0, r0+n) (n <= 32) of sample b (T, U, first row o), one row
// per stage of the warp's TMA ring; the lane that owns a row also takes the
// row's blank and label logits from the staged copy.  kk counts the ring's
// copies so far (stage kk % ST, phase parity (kk / ST) & 1).
template <typename Tin, int NV>
__device__ bool row_batch_tma(const Params& p, int64_t r0, int n, unsigned char* buf,
                              uint64_t* bars, uint32_t& kk, int b, int T, int U, int64_t o) {
    using E = Elt<Tin>;
    constexpr int ST = main_stages(NV);
    constexpr int EPV = E::kPerVec;
    const int wl = threadIdx.x & 31, sb = p.stage_bytes;
    const Tin* X = static_cast<const Tin*>(p.logits);
    const int V = p.V, nvec = V / EPV;
    const uint32_t rb = (uint32_t)V * sizeof(Tin);
    // This lane's row (lane wl owns row r0 + wl): lattice node and label.
    const unsigned rr = (unsigned)(r0 + wl - o);
    const int W = U + 1;
    const int t = (int)(rr / (unsigned)W), u = (int)(rr - (unsigned)t * W);
    const int y = (wl < n && u < U) ? __ldg(p.targets + (int64_t)b * p.S + u) : -1;
    float myhb = 0.0f, myhy = 0.0f;
    if (wl == 0) {
        fence_proxy_async();
        for (int i = 0; i < min(ST, n); ++i) {
            const uint32_t st = (kk + i) % ST;
            tma_row_load(buf + st * sb, X + lrow_s(p, r0 + i, b, o, W) * (int64_t)V, rb,
                         &bars[st]);
        }
    }
    float myM = 0.0f, mys = 0.0f;
    int ifail = -1;
    for (int g0 = 0; g0 < n; g0 += 8) {
        float lm[8], ls[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            lm[j] = -INFINITY;
            ls[j] = 0.0f;
            const int i = g0 + j;
            if (ifail < 0 && i < n) {
                const uint32_t k = kk + i, st = k % ST;
                if (!mbar_wait(&bars[st], (k / ST) & 1, p.err)) {
                    ifail = i;
                } else {
                    const uint4* rv = reinterpret_cast<const uint4*>(buf + st * sb);
                    uint4 q[NV];
#pragma unroll
                    for (int v = 0; v < NV; ++v)
                        if (wl + 32 * v < nvec) q[v] = rv[wl + 32 * v];
                    if (wl == i) {
                        const Tin* rowp = reinterpret_cast<const Tin*>(buf + st * sb);
                        myhb = E::to_f(rowp[p.blank]);
                        myhy = y >= 0 ? E::to_f(rowp[y]) : 0.0f;
                    }
                    __syncwarp();
                    if (wl == 0 && i + ST < n) {
                        fence_proxy_async();
                        tma_row_load(buf + st * sb,
                                     X + lrow_s(p, r0 + i + ST, b, o, W) * (int64_t)V, rb,
                                     &bars[st]);
                    }
                    row_partial<Tin, NV>(q, nvec, wl, lm[j], ls[j]);
                }
            }
        }
        if (ifail >= 0) break;
        float M, S;
        lse_group8(lm, ls, wl, M, S);
        const float vM = __shfl_sync(0xffffffffu, M, 4 * (wl & 7));
        const float vS = __shfl_sync(0xffffffffu, S, 4 * (wl & 7));
        if ((wl & 24) == g0) {
            myM = vM;
            mys = vS;
        }
    }
    if (ifail >= 0) {   // timeout: wait (bounded) for the copies still in flight
        for (int q = ifail; q < min(ifail + ST, n); ++q)
            mbar_wait(&bars[(kk + q) % ST], ((kk + q) / ST) & 1, p.err);
        return false;
    }
    kk += n;
    if (wl < n) row_finish_at<Tin>(p, r0 + wl, myM, mys, myhb, myhy, t, u, T, U, o);
    return true;
}

// Warp: the exactly-zero rows of its own 32-row slice [r0+s0, r0+s0+n) by
// bulk stores from the zeroed shared buffer (zmask: zero rows of the slice),
// then the non-zero rows list[first], list[first+stride], ... (cnt entries,
// row offsets from r0) of the whole task, fetched through the warp's TMA ring.
// Dealing the task's non-zero rows round-robin keeps the warps balanced: they
// cluster along the alignment path, so a 32-row slice may hold none or all.
template <typename Tin, int NV>
__device__ bool grad_batch_tma(const Params& p, int64_t r0, int s0, uint32_t zmask,
                               const uint16_t* list, int cnt, int first, int stride,
                               const float4* inf, unsigned char* buf, uint64_t* bars,
                               uint32_t& kk, const unsigned char* zbuf, int b, int64_t o,
                               int W) {
    using E = Elt<Tin>;
    constexpr int ST = main_stages(NV);
    constexpr int EPV = E::kPerVec;
    const int wl = threadIdx.x & 31, sb = p.stage_bytes;
    const Tin* X = static_cast<const Tin*>(p.logits);
    Tin* Y = static_cast<Tin*>(p.grad);
    const int V = p.V, nvec = V / EPV;
    const uint32_t rb = (uint32_t)V * sizeof(Tin);
    const float cl = p.clamp * p.scale;
    const bool clip = p.clamp < INFINITY;
    const int vb = p.blank / EPV, eb_i = p.blank % EPV;
    const int my = cnt > first ? (cnt - first + stride - 1) / stride : 0;
    if (wl == 0) {
        uint32_t zm = zmask;
        while (zm) {
            const int a = __ffs(zm) - 1;
            const uint32_t after = ~(zm >> a);
            const int len = after ? __ffs(after) - 1 : 32 - a;
            for (int k = 0; k < len;) {
                // One bulk store per run of rows that are consecutive in memory
                // (in the padded layout a run ends with its lattice row).
                const int64_t rs = r0 + s0 + a + k;
                int nr = min(p.zero_rows, len - k);
                if (p.padded) nr = min(nr, W - (int)((unsigned)(rs - o) % (unsigned)W));
                tma_store(Y + lrow_s(p, rs, b, o, W) * (int64_t)V, zbuf, (uint32_t)nr * rb);
                k += nr;
            }
            zm &= len >= 32 ? 0u : ~(((1u << len) - 1u) << a);
        }
        tma_store_commit();
        fence_proxy_async();
        for (int i = 0; i < min(ST, my); ++i) {
            const uint32_t st = (kk + i) % ST;
            tma_row_load(buf + st * sb,
                         X + lrow_s(p, r0 + list[first + i * stride], b, o, W) * (int64_t)V, rb,
                         &bars[st]);
        }
    }
    for (int i = 0; i < my; ++i) {
        const int row = list[first + i * stride];
        const float4 in = inf[row];
        const float w2 = in.x, eb = in.y, ey = in.z;
        const int y = __float_as_int(in.w);
        const int vy = y >= 0 ? y / EPV : -1, ey_i = y >= 0 ? y % EPV : 0;
        const uint32_t k = kk + i, st = k % ST;
        if (!mbar_wait(&bars[st], (k / ST) & 1, p.err)) {
            // Timeout: wait (bounded) for the copies still in flight.
            for (int q = i + 1; q < min(i + ST, my); ++q)
                mbar_wait(&bars[(kk + q) % ST], ((kk + q) / ST) & 1, p.err);
            return false;
        }
        const uint4* rv = reinterpret_cast<const uint4*>(buf + st * sb);
        uint4* ov = reinterpret_cast<uint4*>(Y + lrow_s(p, r0 + row, b, o, W) * (int64_t)V);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int vi = wl + 32 * v;
            if (vi >= nvec) continue;
            float g[EPV];
            {
                float x[EPV];
                E::unpack(rv[vi], x);
#pragma unroll
                for (int e = 0; e < EPV; ++e) g[e] = ex2(fmaf(x[e], kLog2e, w2));
            }
            if (vi == vb) {
#pragma unroll
                for (int e = 0; e < EPV; ++e)
                    if (e == eb_i) g[e] -= eb;
            }
            if (vi == vy) {
#pragma unroll
                for (int e = 0; e < EPV; ++e)
                    if (e == ey_i) g[e] -= ey;
            }
            if (clip) {
#pragma unroll
                for (int e = 0; e < EPV; ++e) g[e] = fminf(fmaxf(g[e], -cl), cl);
            }
            __stcs(ov + vi, E::pack(g));
        }
        __syncwarp();
        if (wl == 0 && i + ST < my) {
            fence_proxy_async();
            tma_row_load(
                buf + st * sb,
                X + lrow_s(p, r0 + list[first + (i + ST) * stride], b, o, W) * (int64_t)V, rb,
                &bars[st]);
        }
    }
    kk += my;
    return true;
}

// Warp: gradient rows without staging (log-softmax off: nothing is read).
template <typename Tin, int G, bool VEC, bool FUSED>
__device__ void grad_batch_plain(const Params& p, int64_t r0, int n, const float4* inf, int b,
                                 int64_t o, int W) {
    using E = Elt<Tin>;
    constexpr int NG = 32 / G;
    const Tin* X = static_cast<const Tin*>(p.logits);
    Tin* Y = static_cast<Tin*>(p.grad);
    const int V = p.V;
    const int wl = threadIdx.x & 31, lane = wl & (G - 1), grp = wl / G;
    const float cl = p.clamp * p.scale;
    const bool clip = p.clamp < INFINITY;
    for (int it = grp; it < n; it += NG) {
        const float4 in = inf[it];
        const bool zero = in.x == -INFINITY;
        const float w2 = in.x, eb = in.y, ey = in.z;
        const int y = __float_as_int(in.w);
        const int64_t lr = lrow_s(p, r0 + it, b, o, W);
        const Tin* row = X + lr * (int64_t)V;
        Tin* out = Y + lr * (int64_t)V;
        if (VEC) {
            constexpr int EPV = E::kPerVec;
            const int nvec = V / EPV;
            const uint4* rv = reinterpret_cast<const uint4*>(row);
            uint4* ov = reinterpret_cast<uint4*>(out);
            for (int vi = lane; vi < nvec; vi += G) {
                float x[EPV], g[EPV];
                if (FUSED && !zero) E::unpack(__ldcs(rv + vi), x);
#pragma unroll
                for (int e = 0; e < EPV; ++e) {
                    const int k = vi * EPV + e;
                    float gv = (FUSED && !zero) ? ex2(fmaf(x[e], kLog2e, w2)) : 0.0f;
                    if (k == p.blank) gv -= eb;
                    if (k == y) gv -= ey;
                    g[e] = clip ? fminf(fmaxf(gv, -cl), cl) : gv;
                }
                __stcs(ov + vi, E::pack(g));
            }
        } else {
            for (int k = lane; k < V; k += G) {
                float gv = (FUSED && !zero) ? ex2(fmaf(E::to_f(row[k]), kLog2e, w2)) : 0.0f;
                if (k == p.blank) gv -= eb;
                if (k == y) gv -= ey;
                out[k] = E::from_f(clip ? fminf(fmaxf(gv, -cl), cl) : gv);
            }
        }
    }
}

// DP task: the sample's forward and backward recursions on this CTA's warps.
__device__ __noinline__ void dp_task(const Params& p, int b, int4* smem, float2* xch) {
    Samp c;
    c.b = b;
    c.T = __ldg(p.Tl + b);
    c.U = __ldg(p.Ul + b);
    c.W = c.U + 1;
    c.D = c.T + c.U;
    c.off = __ldcg(p.off + b);
    // The persistent kernel is launched only when every lattice's DP fits its
    // shared memory, i.e. at most 2 columns per lane (W <= 256).
    const int J = dp_jclass(dp_slots(c.W));
    if (J == 1) dp_run<1>(p, c, smem, xch);
    else if (J == 2) dp_run<2>(p, c, smem, xch);
    else if (threadIdx.x == 0) atomicOr(p.err, ERR_INTERNAL);
}

// Runs DP(b) on the calling CTA if nobody has claimed it yet (CTA-uniform).
__device__ __forceinline__ void run_dp_and_signal(const Params& p, int b, int4* smem, float2* xch,
                                                  int trace_slot, int tid) {
    const uint64_t t0 = (p.trace && tid == 0) ? global_ns() : 0;
    dp_task(p, b, smem, xch);
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        atomicExch(&p.dpdone[b], 1);
        if (p.trace) trace_task(p, trace_slot, TASK_DP | (b << 2), t0);
    }
}

// NV > 0: log-softmax in kernel, rows staged by TMA (NV vectors per lane).
// NV == 0: log-softmax off, rows gathered (2 elements) and gradients written
// with G lanes per row (VEC: 16-byte rows).
//
// Roles.  CTAs on the first n_dp_sms SMs (by %smid) are DP workers: they take
// samples by ticket in DP order, wait for the sample's row chunks and run its
// recursions, undisturbed by the streaming warps that would otherwise share
// their SM.  All other CTAs stream: row chunks, then gradient chunks.  A
// gradient chunk whose DP nobody has started yet runs that DP itself, so
// progress never depends on where CTAs land.
__device__ void finalize_block(const Params& p);

template <typename Tin, int NV, int G, bool VEC>
__device__ __forceinline__ void main_body(const Params& p) {
    constexpr int ST = main_stages(NV > 0 ? NV : 1);
    extern __shared__ __align__(128) unsigned char smem_raw[];
    __shared__ uint64_t bars_all[8 * ST];
    __shared__ float4 s_info[kTaskRows];
    __shared__ uint16_t s_nz[kTaskRows];
    __shared__ int s_cnt[8];
    __shared__ float2 xch[2 * kDpWarps * kXch];
    __shared__ int s_task, s_go;
    // Set by the preparation before the grid barrier; read through L2 because
    // the preparation ran inside this kernel (as are the offsets, order and
    // task list: none of them is read through the read-only cache here).
    if (__ldcg(p.err) & (ERR_LENGTH | ERR_ROWS | ERR_TARGET)) return;
    const int tid = threadIdx.x, wid = tid >> 5, wl = tid & 31;
    int4* dpsmem = reinterpret_cast<int4*>(smem_raw);
    const int ntasks = __ldcg(p.err + 2);

    if (smid() < p.n_dp_sms) {
        for (;;) {
            if (tid == 0) {
                const int i = atomicAdd(&p.err[3], 1);
                int go = 0;
                if (i < p.B) {
                    const int b = __ldcg(p.order + i);
                    s_task = b;
                    // Wait for the sample's rows unless a streaming CTA took the DP.
                    for (int k = 0; k < kSpinLimit; ++k) {
                        if (ld_acquire(&p.dpclaim[b])) break;
                        if (ld_acquire(&p.rdone[b]) >= __ldcg(p.rtasks + b)) {
                            go = atomicCAS(&p.dpclaim[b], 0, 1) == 0;
                            break;
                        }
                        if (ld_acquire(p.err) & ERR_TIMEOUT) break;
                        __nanosleep(256);
                        if (k == kSpinLimit - 1) report_timeout(p.err, 2, b);
                    }
                    go = go ? 1 : 2;   // 1: run it, 2: skip this sample
                }
                s_go = go;
            }
            __syncthreads();
            const int go = s_go, b = s_task;
            __syncthreads();
            if (go == 0) break;
            if (go == 1) {
                __threadfence();
                run_dp_and_signal(p, b, dpsmem, xch, ntasks + b, tid);
            }
        }
        return;
    }

    unsigned char* buf = smem_raw + (size_t)wid * ST * p.stage_bytes;
    uint64_t* bars = bars_all + wid * ST;
    const unsigned char* zbuf = smem_raw + p.zero_off;
    if (NV > 0) {
        const int zn = p.zero_rows * p.V * (int)sizeof(Tin) / 16;
        for (int i = tid; i < zn; i += blockDim.x)
            reinterpret_cast<uint4*>(smem_raw + p.zero_off)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async();   // generic writes before the bulk stores read them
        __syncthreads();
    }
    if (NV > 0 && wl == 0) {
#pragma unroll
        for (int st = 0; st < ST; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    uint32_t kk = 0;   // this warp's TMA ring position
    for (;;) {
        // Every branch below is taken by the whole CTA: decisions that depend on
        // global state are made by thread 0 and broadcast through shared memory.
        if (tid == 0) {
            s_task = atomicAdd(&p.err[1], 1);
            s_go = !(ld_acquire(p.err) & ERR_TIMEOUT);
        }
        __syncthreads();
        const int t = s_task;
        const bool go = s_go;
        __syncthreads();
        if (t >= ntasks || !go) break;
        const int4 tk = __ldcg(p.tasks + 2 * t), tc = __ldcg(p.tasks + 2 * t + 1);
        const int kind = tk.x & 3, b = tk.x >> 2, n = tk.z;
        const int64_t o_b = (int64_t)(uint32_t)tc.z | ((int64_t)tc.w << 32);
        const int W_b = tc.x + 1;
        const int64_t r0 = o_b + tk.y;
        const uint64_t t_start = (p.trace && tid == 0) ? global_ns() : 0;
        if (kind == TASK_ROW) {
            if (NV > 0) fence_proxy_async();   // smem may have been a DP ring
            const int per = (n + 7) >> 3;   // rows per warp: 32 for a full task
            const int64_t rw = r0 + per * wid;
            const int nw = min(per, n - per * wid);
            if (nw > 0) {
                if (NV > 0) {
                    row_batch_tma<Tin, (NV > 0 ? NV : 1)>(p, rw, nw, buf, bars, kk, b, tk.w,
                                                          tc.x, o_b);
                } else if (flat_rows(p.V, sizeof(Tin), p.fused)) {
                    const Tin* X = static_cast<const Tin*>(p.logits);
                    if (p.padded) {
                        float M = 0.0f, s = 0.0f;
                        if (wl < nw) {
                            flat_row_stats<Tin>(X + lrow_s(p, rw + wl, b, o_b, W_b) * (int64_t)p.V,
                                                p.V, M, s);
                            row_finish<Tin>(p, rw + wl, M, s);
                        }
                    } else {
                        const Tin* rows = flat_stage<Tin>(
                            X, rw, nw, p.V,
                            smem_raw + (size_t)wid * flat_warp_bytes(p.V, sizeof(Tin)), wl);
                        if (wl < nw) {
                            // The sample is the task's, and the blank and label
                            // log-probabilities are in the staged row.
                            const Tin* row = rows + (int64_t)wl * p.V;
                            float M, s;
                            flat_row_stats<Tin>(row, p.V, M, s);
                            const int64_t r = rw + wl;
                            const unsigned rr = (unsigned)(r - o_b);
                            const int t = (int)(rr / (unsigned)W_b), u = (int)(rr - (unsigned)t * W_b);
                            const int U = W_b - 1;
                            const float hb = Elt<Tin>::to_f(row[p.blank]);
                            const float hy =
                                u < U ? Elt<Tin>::to_f(row[__ldg(p.targets + (int64_t)b * p.S + u)])
                                      : 0.0f;
                            row_finish_at<Tin>(p, r, M, s, hb, hy, t, u, tk.w, U, o_b);
                        }
                    }
                } else if (p.fused) {
                    // Rows that are not 16-byte vectors: G-lane groups reduce
                    // the rows (as the per-stage row kernel does), each row's
                    // statistics handed to its lane.
                    constexpr int NG = 32 / G;
                    const int lane = wl & (G - 1), grp = wl / G;
                    const unsigned gm = group_mask<G>();
                    float myM = 0.0f, mys = 0.0f;
                    for (int it = 0; it < G; ++it) {
                        const int ri = it * NG + grp;
                        float M = -INFINITY, s = 0.0f;
                        if (ri < nw)
                            row_stats_stream<Tin, G, VEC>(
                                static_cast<const Tin*>(p.logits) +
                                    lrow_s(p, rw + ri, b, o_b, W_b) * (int64_t)p.V,
                                p.V, lane, gm, M, s);
                        hand_over<G>(it, wl, M, s, myM, mys);
                    }
                    if (wl < nw) row_finish<Tin>(p, rw + wl, myM, mys);
                } else if (wl < nw) {
                    row_finish<Tin>(p, rw + wl, 0.0f, 1.0f);
                }
            }
            __threadfence();
            __syncthreads();
            if (tid == 0) atomicAdd(&p.rdone[b], 1);
            if (p.trace && tid == 0) trace_task(p, t, tk.x, t_start);
            continue;
        }
        // Gradient chunk: its sample's DP must be done (or be run here).
        if (tid == 0) {
            int mode = 0;   // 0: error, 1: DP done, 2: run the DP here
            for (int k = 0; k < kSpinLimit; ++k) {
                if (ld_acquire(&p.dpdone[b])) {
                    mode = 1;
                    break;
                }
                if (ld_acquire(&p.rdone[b]) >= __ldcg(p.rtasks + b) &&
                    ld_acquire(&p.dpclaim[b]) == 0 && atomicCAS(&p.dpclaim[b], 0, 1) == 0) {
                    mode = 2;
                    break;
                }
                if (ld_acquire(p.err) & ERR_TIMEOUT) break;
                __nanosleep(128);
                if (k == kSpinLimit - 1) report_timeout(p.err, 3, b);
            }
            s_go = mode;
        }
        __syncthreads();
        const int mode = s_go;
        __syncthreads();
        __threadfence();
        if (mode == 0) continue;   // uniform; the next iteration sees the error and stops
        if (mode == 2) {
            run_dp_and_signal(p, b, dpsmem, xch, ntasks + b, tid);
            __syncthreads();
        }
        if (NV > 0) fence_proxy_async();   // smem may have been a DP ring
        if (tid < n) s_info[tid] = combine_row(p, r0 + tid, b);
        __syncthreads();
        const int nw = min(32, n - 32 * wid);
        if (NV > 0) {
            // Compact the task's non-zero rows (in row order) for round-robin dealing.
            const bool nz = tid < n && s_info[tid].x != -INFINITY;
            const uint32_t bal = __ballot_sync(0xffffffffu, nz);
            if (wl == 0) s_cnt[wid] = __popc(bal);
            __syncthreads();
            int before = 0, cnt = 0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int ck = s_cnt[k];
                before += k < wid ? ck : 0;
                cnt += ck;
            }
            if (nz) s_nz[before + __popc(bal & ((1u << wl) - 1u))] = (uint16_t)tid;
            __syncthreads();
            const uint32_t zmask = nw > 0 ? ~bal & (nw >= 32 ? 0xffffffffu : ((1u << nw) - 1u)) : 0u;
            grad_batch_tma<Tin, (NV > 0 ? NV : 1)>(p, r0, 32 * wid, zmask, s_nz, cnt, wid, 8,
                                                  s_info, buf, bars, kk, zbuf, b, o_b, W_b);
        } else if (nw > 0) {
            if (flat_rows(p.V, sizeof(Tin), p.fused) && !p.padded)
                flat_grad<Tin>(p, r0 + 32 * wid, nw, wl, [&](int i) { return s_info[32 * wid + i]; });
            else if (p.fused)
                grad_batch_plain<Tin, G, VEC, true>(p, r0 + 32 * wid, nw, s_info + 32 * wid, b, o_b,
                                                    W_b);
            else
                grad_batch_plain<Tin, G, VEC, false>(p, r0 + 32 * wid, nw, s_info + 32 * wid, b,
                                                     o_b, W_b);
        }
        if (p.trace) {
            __syncthreads();
            if (tid == 0) trace_task(p, t, tk.x, t_start);
        }
    }
    // Zero-row bulk stores read the shared buffer until they complete.
    if (NV > 0 && wl == 0) tma_store_wait_all();
}


// The last CTA to finish runs the loss check and reduction (no separate
// finalize launch): every CTA publishes its writes and counts itself out.
// The call's preparation runs first on CTA 0 (no separate launch); a grid-wide
// barrier of the cooperative launch then releases every CTA.
template <typename Tin, int NV, int G, bool VEC>
__global__ void __launch_bounds__(256, 2) k_main(Params p) {
    extern __shared__ __align__(128) unsigned char smem_dyn[];
    if (blockIdx.x == 0)
        prepare_block(p, reinterpret_cast<int64_t*>(smem_dyn),
                      reinterpret_cast<int*>(smem_dyn + sizeof(int64_t) * blockDim.x));
    cooperative_groups::this_grid().sync();
    main_body<Tin, NV, G, VEC>(p);
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&p.err[8], 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (s_last) {
        __threadfence();
        finalize_block(p);
    }
}

// ---------------------------------------------------------------- finalize
// Loss check, reduction and status, by one CTA of 256 threads (every thread).
__device__ void finalize_block(const Params& p) {
    __shared__ double part[256];
    __shared__ int errs;
    const int tid = threadIdx.x;
    if (tid == 0) errs = __ldcg(p.err);
    __syncthreads();
    const bool ok_in = (errs & (ERR_LENGTH | ERR_ROWS | ERR_TARGET | ERR_TIMEOUT | ERR_INTERNAL)) == 0;
    double s = 0.0;
    if (ok_in) {
        for (int b = tid; b < p.B; b += blockDim.x) {
            const double la = __ldcg(p.lossa + b), lb = __ldcg(p.lossb + b);
            if (!(fabs(la - lb) <= 1e-3 * fmax(1.0, fabs(la)))) atomicOr(&errs, ERR_MISMATCH);
            s += la;
        }
    }
    part[tid] = s;
    __syncthreads();
    for (int o = blockDim.x / 2; o > 0; o >>= 1) {
        if (tid < o) part[tid] += part[tid + o];
        __syncthreads();
    }
    if (tid == 0) {
        if (ok_in && p.loss_red)
            p.loss_red[0] = (float)(p.red == RNNT_RED_MEAN ? part[0] / p.B : part[0]);
        int st = RNNT_OK;
        if (errs & (ERR_LENGTH | ERR_ROWS | ERR_TARGET)) st = RNNT_INVALID_VALUE;
        else if (errs & ERR_TIMEOUT) st = RNNT_TIMEOUT;
        else if (errs & ERR_INTERNAL) st = RNNT_LAUNCH_FAILED;
        else if (errs & (ERR_MISMATCH | ERR_NONFINITE)) st = RNNT_LOSS_MISMATCH;
        *p.err = errs;
        if (p.status) *p.status = st;
    }
}

__global__ void __launch_bounds__(256) k_finalize(Params p) { finalize_block(p); }

// ---------------------------------------------------------------- multi-blank
// Multi-blank transducer (ESPnet compute_multiblank_grad_kernel docs): besides
// the one-frame blank, big blank i (output bb_id[i]) moves bb_dur[i] frames.
// A path ends when a blank-type step reaches frame T with all U labels out.
//
// k_dp_mb: one CTA per (sample, direction), blockIdx.y = 0 forward (alpha),
// 1 backward (beta).  Thread u owns lattice column u and walks the
// anti-diagonals, one node per diagonal.  Only the label arc crosses columns:
// its product goes through a double-buffered exchange in shared memory, one
// barrier per diagonal.  Blank and big-blank arcs stay in the column: each
// thread keeps its column's last kMbRing values in a private shared-memory
// ring (slot t mod kMbRing), so a big blank of up to kMbRing frames needs no
// extra barrier.  Extended-range arithmetic as in the standard recursions;
// every transition probability is scaled by bb_c = e^-sigma.
constexpr int kMbRing = RNNT_MAX_BIG_BLANK_DURATION;
static_assert((kMbRing & (kMbRing - 1)) == 0, "ring slots are t mod a power of two");

// a += x * p * c without renormalising (the caller renormalises once per
// step: xf_add aligns unnormalised mantissas exactly).
__device__ __forceinline__ void xf_mac_raw(float& am, int& ae, float xm, int xe, float pm, int pe,
                                           float c) {
    xf_add<false>(am, ae, xm * (pm * c), xe + pe, am, ae);
}

__device__ __forceinline__ void xf_mac(float& am, int& ae, float xm, int xe, float pm, int pe,
                                       float c) {
    // a += x * p * c
    float m = xm * pm * c;
    int e = xe + pe;
    xf_norm(m, e);
    xf_add(am, ae, m, e, am, ae);
}

template <int NT>   // block size bound: 256 (lattices of up to 256 columns) or 1024
__global__ void __launch_bounds__(NT) k_dp_mb(Params p) {
    if (*p.err) return;
    extern __shared__ float2 mb_smem[];
    const int nthr = blockDim.x, u = threadIdx.x;
    float2* ring = mb_smem;                          // [kMbRing][nthr]: {m, e bits}
    float2* xch = mb_smem + (size_t)kMbRing * nthr;  // [2][nthr]
    // [kMbRing][nthr]: node index of this column's node at frame t (slot t mod
    // kMbRing), for the big blanks' source nodes.
    int* iring = reinterpret_cast<int*>(mb_smem + (size_t)(kMbRing + 2) * nthr);
    const int b = blockIdx.x;
    const int T = __ldg(p.Tl + b), U = __ldg(p.Ul + b), W = U + 1, D = T + U, mTW = min(T, W);
    const int64_t o = __ldcg(p.off + b);
    const bool col = u < W;
    const float c = p.bb_c;
    const float2 zero = make_float2(0.0f, __int_as_float(kZeroExp));
    const bool fwd = blockIdx.y == 0;
    // Records of this column's node at the next diagonal, loaded one diagonal
    // ahead: its transition record and the big-blank probabilities it needs
    // (forward: of the big blanks' source nodes (t - dur, u); backward: its own).
    int4 ed_n = make_int4(0, 0, 0, 0);
    int2 q_n[RNNT_MAX_BIG_BLANKS];
#pragma unroll
    for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) q_n[i] = make_int2(0, 0);
    // Node index (in the sample) of this column's node at the fetched frame,
    // stepped from frame to frame: idx(t+1,u) = idx(t,u) + len(d) + 1 - [d >= U]
    // (d = t + u, len(d) the length of anti-diagonal d).
    int fi = 0;
    auto step_len = [&](int dd) { return min(min(dd + 1, mTW), D - dd) + 1 - (dd >= U ? 1 : 0); };
    auto fetch = [&](int t) {
        if (!(col && t >= 0 && t < T)) return;
        if (fwd) fi = t == 0 ? (int)node_index(0, u, T, U) : fi + step_len(t - 1 + u);
        else fi = t == T - 1 ? (int)node_index(T - 1, u, T, U) : fi - step_len(t + u);
        ed_n = __ldcg(p.edge + o + fi);
#pragma unroll
        for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) {
            if (i >= p.K) break;
            const int ts = fwd ? t - p.bb_dur[i] : t;
            const int si = fwd ? iring[(ts & (kMbRing - 1)) * nthr + u] : fi;
            q_n[i] = ts >= 0 ? __ldcg(p.pbb + (int64_t)i * p.rows + o + si) : make_int2(0, 0);
        }
        if (fwd) iring[(t & (kMbRing - 1)) * nthr + u] = fi;
    };
    if (fwd) {
        float bm = 0.0f;   // alpha(t-1,u) p_blank(t-1,u) c: this column's blank outflow
        int be = kZeroExp;
        fetch(-u);
        for (int d = 0; d < D; ++d) {
            const int t = d - u;
            const int4 ed = ed_n;
            const int ni = fi;   // node index of (t, u)
            int2 q[RNNT_MAX_BIG_BLANKS];
#pragma unroll
            for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) q[i] = q_n[i];
            fetch(t + 1);
            float2 out = zero;
            if (col && t >= 0 && t < T) {
                float am;
                int ae;
                if (t == 0 && u == 0) {
                    am = 1.0f;
                    ae = 0;
                } else {
                    // Two accumulators (blank + odd big blanks, label + even
                    // ones) halve the dependent chain; one renormalisation.
                    am = bm;
                    ae = be;
                    float a2 = 0.0f;
                    int e2 = kZeroExp;
                    if (u > 0) {
                        const float2 v = xch[((d - 1) & 1) * nthr + u - 1];
                        a2 = v.x;
                        e2 = __float_as_int(v.y);
                    }
#pragma unroll
                    for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) {
                        if (i >= p.K) break;
                        const int t0 = t - p.bb_dur[i];
                        if (t0 < 0) continue;
                        const float2 a = ring[(t0 & (kMbRing - 1)) * nthr + u];
                        if (i & 1)
                            xf_mac_raw(am, ae, a.x, __float_as_int(a.y), __int_as_float(q[i].x),
                                       q[i].y - kEdgeBias, c);
                        else
                            xf_mac_raw(a2, e2, a.x, __float_as_int(a.y), __int_as_float(q[i].x),
                                       q[i].y - kEdgeBias, c);
                    }
                    xf_add<true>(am, ae, a2, e2, am, ae);
                }
                p.alpha[o + ni] = make_int2(__float_as_int(am), ae);
                ring[(t & (kMbRing - 1)) * nthr + u] = make_float2(am, __int_as_float(ae));
                // Outflows (blank to (t+1,u), label to (t,u+1)); their mantissas
                // stay below 4 and are renormalised by the adds they enter.
                bm = am * (__int_as_float(ed.x) * c);
                be = ae + ed.y - kEdgeBias;
                const float ym = am * (__int_as_float(ed.z) * c);
                const int ye = ae + ed.w - kEdgeBias;
                out = make_float2(ym, __int_as_float(ye));
            } else {
                bm = 0.0f;
                be = kZeroExp;
            }
            xch[(d & 1) * nthr + u] = out;
            __syncthreads();
        }
        if (u == U) {
            // P(y|x): the blank from (T-1,U) plus every big blank that ends at frame T.
            float pm = bm;
            int pe = be;
            for (int i = 0; i < p.K; ++i) {
                const int t0 = T - p.bb_dur[i];
                if (t0 < 0) continue;
                const float2 a = ring[(t0 & (kMbRing - 1)) * nthr + u];
                const int2 q = __ldcg(p.pbb + (int64_t)i * p.rows + o + node_index(t0, u, T, U));
                xf_mac(pm, pe, a.x, __float_as_int(a.y), __int_as_float(q.x), q.y - kEdgeBias, c);
            }
            p.pm[b] = pm;
            p.pe[b] = pe;
            const double ll2 = (double)pe + log2((double)pm);
            p.lossa[b] = -ll2 * kLn2d;
            p.loss[b] = (float)(-ll2 * kLn2d);
        }
    } else {
        float qm = 0.0f;   // beta(t+1,u): this column's previous node
        int qe = kZeroExp;
        fetch(D - 1 - u);
        for (int d = D - 1; d >= 0; --d) {
            const int t = d - u;
            const int4 ed = ed_n;
            const int ni = fi;   // node index of (t, u)
            int2 q[RNNT_MAX_BIG_BLANKS];
#pragma unroll
            for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) q[i] = q_n[i];
            fetch(t - 1);
            float2 out = zero;
            if (col && t >= 0 && t < T) {
                // Two accumulators (blank + odd big blanks, label + even ones).
                float m = 0.0f, m2 = 0.0f;
                int e = kZeroExp, e2 = kZeroExp;
                if (t + 1 < T) xf_mac_raw(m, e, qm, qe, __int_as_float(ed.x), ed.y - kEdgeBias, c);
                else if (u == U) xf_mac_raw(m, e, 1.0f, 0, __int_as_float(ed.x), ed.y - kEdgeBias, c);
                if (u < U) {
                    const float2 v = xch[((d + 1) & 1) * nthr + u + 1];
                    xf_mac_raw(m2, e2, v.x, __float_as_int(v.y), __int_as_float(ed.z),
                               ed.w - kEdgeBias, c);
                }
#pragma unroll
                for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) {
                    if (i >= p.K) break;
                    const int t1 = t + p.bb_dur[i];
                    if (t1 > T || (t1 == T && u != U)) continue;
                    float am2 = 1.0f;
                    int ae2 = 0;
                    if (t1 < T) {
                        const float2 a = ring[(t1 & (kMbRing - 1)) * nthr + u];
                        am2 = a.x;
                        ae2 = __float_as_int(a.y);
                    }
                    if (i & 1) xf_mac_raw(m, e, am2, ae2, __int_as_float(q[i].x), q[i].y - kEdgeBias, c);
                    else xf_mac_raw(m2, e2, am2, ae2, __int_as_float(q[i].x), q[i].y - kEdgeBias, c);
                }
                xf_add<true>(m, e, m2, e2, m, e);
                p.beta[o + ni] = make_int2(__float_as_int(m), e);
                out = make_float2(m, __int_as_float(e));
                ring[(t & (kMbRing - 1)) * nthr + u] = out;
                qm = m;
                qe = e;
            } else {
                qm = 0.0f;
                qe = kZeroExp;
            }
            xch[(d & 1) * nthr + u] = out;
            __syncthreads();
        }
        if (u == 0) p.lossb[b] = -((double)qe + log2((double)qm)) * kLn2d;
    }
}

template <typename Tin, bool VEC>
__global__ void __launch_bounds__(256) k_grad_mb(Params p) {
    if (*p.err) return;
    using E = Elt<Tin>;
    const Tin* X = static_cast<const Tin*>(p.logits);
    Tin* Y = static_cast<Tin*>(p.grad);
    const int V = p.V, wl = threadIdx.x & 31;
    const int64_t nr = nodes(p), nbatch = (nr + 31) / 32;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x / 32);
    const float cl = p.clamp * p.scale;
    const bool clip = p.clamp < INFINITY;
    constexpr unsigned F = 0xffffffffu;
    for (int64_t bt = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; bt < nbatch;
         bt += nwarps) {
        const int64_t r0 = bt * 32;
        const int n = (int)min((int64_t)32, nr - r0);
        MbRec mine;
        if (wl < n) mine = mb_record(p, r0 + wl, find_sample(p.off, p.B, r0 + wl));
        for (int it = 0; it < n; ++it) {
            const float w2 = __shfl_sync(F, mine.w2, it), eb = __shfl_sync(F, mine.eb, it);
            const float ey = __shfl_sync(F, mine.ey, it);
            const int y = __shfl_sync(F, mine.y, it);
            const bool zero = __shfl_sync(F, (int)mine.zero, it) != 0;
            const int64_t lr = __shfl_sync(F, mine.lr, it);
            float ebb[RNNT_MAX_BIG_BLANKS];
#pragma unroll
            for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i)
                ebb[i] = i < p.K ? __shfl_sync(F, mine.ebb[i], it) : 0.0f;
            const Tin* row = X + lr * (int64_t)V;
            Tin* out = Y + lr * (int64_t)V;
            // The element's gradient from its softmax term gk (0 when not fused).
            auto finish = [&](int k, float gk) -> float {
                if (zero) return 0.0f;
                if (k == p.blank) gk -= eb * p.scale;
                if (k == y) gk -= ey * p.scale;
#pragma unroll
                for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i)
                    if (i < p.K && k == p.bb_id[i]) gk -= ebb[i] * p.scale;
                return clip ? fminf(fmaxf(gk, -cl), cl) : gk;
            };
            if (VEC) {
                constexpr int EPV = E::kPerVec;
                const uint4* rv = reinterpret_cast<const uint4*>(row);
                uint4* ov = reinterpret_cast<uint4*>(out);
                for (int vi = wl; vi < V / EPV; vi += 32) {
                    float g[EPV];
                    if (p.fused && !zero) {
                        float x[EPV];
                        E::unpack(__ldcs(rv + vi), x);
#pragma unroll
                        for (int e = 0; e < EPV; ++e) g[e] = ex2(fmaf(x[e], kLog2e, w2));
                    } else {
#pragma unroll
                        for (int e = 0; e < EPV; ++e) g[e] = 0.0f;
                    }
                    // Only a vector that holds an arc's output needs the subtractions.
                    const int k0 = vi * EPV;
                    bool special = (unsigned)(p.blank - k0) < (unsigned)EPV ||
                                   (unsigned)(y - k0) < (unsigned)EPV;
                    for (int i = 0; i < p.K; ++i)
                        special |= (unsigned)(p.bb_id[i] - k0) < (unsigned)EPV;
                    if (special) {
#pragma unroll
                        for (int e = 0; e < EPV; ++e) g[e] = finish(k0 + e, g[e]);
                    } else if (clip && !zero) {
#pragma unroll
                        for (int e = 0; e < EPV; ++e) g[e] = fminf(fmaxf(g[e], -cl), cl);
                    } else if (zero) {
#pragma unroll
                        for (int e = 0; e < EPV; ++e) g[e] = 0.0f;
                    }
                    __stcs(ov + vi, E::pack(g));
                }
            } else {
                for (int k = wl; k < V; k += 32) {
                    const float gk =
                        (p.fused && !zero) ? ex2(fmaf(E::get(row, k), kLog2e, w2)) : 0.0f;
                    out[k] = E::from_f(finish(k, gk));
                }
            }
        }
    }
}

// ---------------------------------------------------------------- self-test
// The bounded-wait path, exercised without any fault: one warp waits, through
// the same helper as the row rings, on an mbarrier that nothing ever
// completes; the wait gives up after `limit` polls, records the timeout in an
// error word the way every kernel here does, and the kernel reports
// RNNT_TIMEOUT in status.  Nothing is left in flight.
__global__ void __launch_bounds__(32) k_selftest_wait(int32_t* status, int limit) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int32_t err[16];
    const int wl = threadIdx.x;
    if (wl < 16) err[wl] = 0;
    if (wl == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    mbar_wait(&bar, 0, err, limit);
    __syncwarp();
    if (wl == 0) *status = (err[0] & ERR_TIMEOUT) ? RNNT_TIMEOUT : RNNT_OK;
}

// ---------------------------------------------------------------- padding
// Padded layout: zero gradient rows outside every lattice (t >= T_b or
// u > U_b), one warp per row; rows inside a lattice are left to the gradient
// pass.  Reads only the lengths, so it needs nothing from the preparation.
template <typename Tin>
__global__ void __launch_bounds__(256) k_pad_zero(Params p) {
    const int64_t per = (int64_t)p.maxT * p.maxW;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x / 32);
    const int lane = threadIdx.x & 31;
    const int64_t rb = (int64_t)p.V * sizeof(Tin);
    for (int64_t R = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; R < p.rows; R += nw) {
        const int b = (int)(R / per);
        const int64_t q = R - (int64_t)b * per;
        const int t = (int)(q / p.maxW), u = (int)(q - (int64_t)t * p.maxW);
        if (t < __ldg(p.Tl + b) && u <= __ldg(p.Ul + b)) continue;
        char* row = static_cast<char*>(p.grad) + R * rb;
        if (rb % 16 == 0) {
            for (int64_t k = lane; k < rb / 16; k += 32)
                __stcs(reinterpret_cast<uint4*>(row) + k, make_uint4(0, 0, 0, 0));
        } else {
            for (int k = lane; k < p.V; k += 32) reinterpret_cast<Tin*>(row)[k] = Elt<Tin>::from_f(0.0f);
        }
    }
}

// ---------------------------------------------------------------- grad scale
// hdr: the call's workspace header; hdr[12] = rows per sample slot of the
// padded layout, 0 for the compact one.
template <typename Tin>
__global__ void __launch_bounds__(256) k_scale(void* grad, int64_t rows, int V, int B,
                                               const int64_t* off, const int32_t* hdr,
                                               const float* factors, int per_sample) {
    if (!per_sample && factors[0] == 1.0f) return;
    using E = Elt<Tin>;
    Tin* G = static_cast<Tin*>(grad);
    const int64_t ng = (int64_t)gridDim.x * (blockDim.x / 32);
    const int lane = threadIdx.x & 31;
    const int64_t per = hdr[12];
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; r < rows; r += ng) {
        const int b = per > 0 ? (int)min(r / per, (int64_t)B - 1) : find_sample(off, B, r);
        const float f = per_sample ? factors[b] : factors[0];
        if (f == 1.0f) continue;
        Tin* row = G + r * (int64_t)V;
        for (int k = lane; k < V; k += 32) row[k] = E::from_f(E::to_f(row[k]) * f);
    }
}

// ---------------------------------------------------------------- host side
// Runs f(T{}) with T the storage type of dt (float, __half or __nv_bfloat16).
template <typename F>
auto with_type(rnnt_dtype_t dt, F&& f) {
    if (dt == RNNT_F32) return f(float{});
    if (dt == RNNT_F16) return f(__half{});
    return f(__nv_bfloat16{});
}
bool valid_dtype(rnnt_dtype_t dt) { return dt == RNNT_F32 || dt == RNNT_F16 || dt == RNNT_BF16; }

int g_num_sms[64];
int g_dp_smem_set[64];

int num_sms(int dev) {
    if (dev < 0 || dev >= 64) return 148;
    if (!g_num_sms[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        g_num_sms[dev] = n;
    }
    return g_num_sms[dev];
}

// DP shared memory of both directions for every lattice width up to S+1
// (the persistent kernel's DP task: one-warp recursions up to 32 *
// kWarpDpMaxJ columns, the multi-warp ones above).
size_t dp_smem_for(int S) {
    size_t best = 0;
    for (int W = 1; W <= S + 1; ++W) {
        const size_t b = W <= 32 * kWarpDpMaxJ ? wdp_smem_bytes(W) : dp_smem_bytes(W);
        if (b > best) best = b;
    }
    return best;
}
// The per-stage DP (one direction per CTA): half the rings, and the table.
size_t dp_smem_dir_for(int S) {
    size_t best = 0;
    for (int W = 1; W <= S + 1; ++W) {
        const size_t b = W <= 32 * kWarpDpMaxJ ? wdp_smem_bytes(W) / 2
                                               : dp_deep_ring_bytes(W) + (size_t)kTabMax * sizeof(int);
        if (b > best) best = b;
    }
    return best;
}
int dp_threads_for(int S) {
    return S + 1 <= 32 * kWarpDpMaxJ ? 32 : 32 * dp_warps(S + 1, kDpWarpsStaged);
}

int grid_for(int64_t work_threads, int sms, int per_sm) {
    const int64_t blocks = (work_threads + 255) / 256;
    const int64_t cap = (int64_t)sms * per_sm;
    return (int)(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

// Resident 256-thread blocks per SM of a kernel (cached per kernel).
// Resident CTAs per SM of `kernel` with 256 threads and `smem` bytes of
// dynamic shared memory; sets the kernel's dynamic shared memory limit to
// exactly `smem` (the limit, not only the launch's request, decides how many
// CTAs a cooperative launch may place on an SM).  Cached per (kernel, smem).
int occupancy(const void* kernel, size_t smem) {
    static const void* keys[128];
    static size_t smems[128];
    static int vals[128];
    static const void* attr_fn[64];
    static size_t attr_val[64];
    // The kernel's current limit (per process; one device's attributes are
    // assumed to match the others').
    int slot = -1;
    for (int i = 0; i < 64; ++i)
        if (attr_fn[i] == kernel || !attr_fn[i]) {
            slot = i;
            break;
        }
    if (slot >= 0 && (attr_fn[slot] != kernel || attr_val[slot] != smem)) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        attr_fn[slot] = kernel;
        attr_val[slot] = smem;
    }
    for (int i = 0; i < 128 && keys[i]; ++i)
        if (keys[i] == kernel && smems[i] == smem) return vals[i];
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, smem) != cudaSuccess || n < 1) {
        cudaGetLastError();
        n = 0;
    }
    for (int i = 0; i < 128 && n > 0; ++i)
        if (!keys[i]) {
            vals[i] = n;
            smems[i] = smem;
            keys[i] = kernel;
            break;
        }
    return n;
}

// Grid-stride launch: never more blocks than are resident at once.
template <typename K>
void launch_gs(K kernel, int64_t work_threads, int sms, cudaStream_t st, const Params& p,
               size_t smem = 0) {
    const int occ = occupancy(reinterpret_cast<const void*>(kernel), smem);
    const int g = grid_for(work_threads, sms, occ > 0 ? occ : 1);
    kernel<<<g, 256, smem, st>>>(p);
}

// Shared memory of the TMA-staged passes: kStages row buffers + barriers per warp.
size_t tma_smem(const Params& p) {
    return (size_t)8 * kStages * p.stage_bytes + (size_t)8 * kStages * sizeof(uint64_t);
}

// Lanes per row of the log-softmax statistics for rows that are not 16-byte
// vectors and at most 1 KB long, on either schedule (the same reduction order,
// so that both give the same bits).
inline int plain_group(int V) { return V >= 256 ? 32 : 8; }

template <typename Tin>
void launch_rows(const Params& p, cudaStream_t st, int sms) {
    const int V = p.V;
    if (!p.fused) {
        k_row_gather<Tin><<<(unsigned)((p.rows + kGatherNodes - 1) / kGatherNodes), 256, 0, st>>>(p);
        return;
    }

    constexpr int EPV = Elt<Tin>::kPerVec;
    const bool vec = ((size_t)V * sizeof(Tin)) % 16 == 0;
    const int nvec = V / EPV;
    const int64_t wt = (p.rows + 31) / 32 * 32;   // one warp per 32-row batch
    if (vec && nvec > 32 && nvec <= 32 * 8) {
        const size_t sm = tma_smem(p);
        if (nvec <= 64) launch_gs(k_row_tma<Tin, 2>, wt, sms, st, p, sm);
        else if (nvec <= 128) launch_gs(k_row_tma<Tin, 4>, wt, sms, st, p, sm);
        else launch_gs(k_row_tma<Tin, 8>, wt, sms, st, p, sm);
        return;
    }
    if (vec && nvec <= 32 * 8) {
        if (nvec <= 4) launch_gs(k_row_regs<Tin, 4, 1>, wt, sms, st, p);
        else if (nvec <= 16) launch_gs(k_row_regs<Tin, 8, 2>, wt, sms, st, p);
        else if (nvec <= 32) launch_gs(k_row_regs<Tin, 16, 2>, wt, sms, st, p);
        else if (nvec <= 64) launch_gs(k_row_regs<Tin, 32, 2>, wt, sms, st, p);
        else if (nvec <= 128) launch_gs(k_row_regs<Tin, 32, 4>, wt, sms, st, p);
        else launch_gs(k_row_regs<Tin, 32, 8>, wt, sms, st, p);
        return;
    }
    if (flat_rows(V, sizeof(Tin), p.fused)) {
        launch_gs(k_row_flat<Tin>, wt, sms, st, p, 8 * flat_warp_bytes(V, sizeof(Tin)));
        return;
    }
    if (!vec && (size_t)V * sizeof(Tin) <= 1024) {
        if (plain_group(V) == 32) launch_gs(k_row_stream<Tin, 32, false>, wt, sms, st, p);
        else launch_gs(k_row_stream<Tin, 8, false>, wt, sms, st, p);
        return;
    }
#define ROWK(G_)                                                                 \
    do {                                                                         \
        if (vec) launch_gs(k_row_stream<Tin, G_, true>, wt, sms, st, p);         \
        else launch_gs(k_row_stream<Tin, G_, false>, wt, sms, st, p);            \
    } while (0)
    if (V >= 512) ROWK(32);
    else if (V >= 128) ROWK(16);
    else if (V >= 32) ROWK(8);
    else ROWK(4);
#undef ROWK
}

// Returns true when the launched kernel also ran the loss check.
template <typename Tin>
bool launch_grad(const Params& p, cudaStream_t st, int sms) {
    const int V = p.V;

    const bool vec = ((size_t)V * sizeof(Tin)) % 16 == 0;
    const int nvec = V / Elt<Tin>::kPerVec;
    if (p.fused && vec && nvec > 32 && nvec <= 32 * 8) {
        const size_t sm = tma_smem(p);
        const int64_t wt = (p.rows + 31) / 32 * 32;
        if (nvec <= 64) launch_gs(k_grad_tma<Tin, 2>, wt, sms, st, p, sm);
        else if (nvec <= 128) launch_gs(k_grad_tma<Tin, 4>, wt, sms, st, p, sm);
        else launch_gs(k_grad_tma<Tin, 8>, wt, sms, st, p, sm);
        return true;
    }
    if (p.info) {   // long rows: records from k_combine
        const int64_t wt = p.rows * 32;
        if (p.fused) {
            if (vec) launch_gs(k_grad_long<Tin, true, true>, wt, sms, st, p);
            else launch_gs(k_grad_long<Tin, false, true>, wt, sms, st, p);
        } else {
            if (vec) launch_gs(k_grad_long<Tin, true, false>, wt, sms, st, p);
            else launch_gs(k_grad_long<Tin, false, false>, wt, sms, st, p);
        }
        return false;
    }
#define GRADK(G_)                                                                      \
    do {                                                                               \
        const int64_t wt = p.rows * G_;                                                \
        if (p.fused) {                                                                 \
            if (vec) launch_gs(k_grad<Tin, G_, true, true>, wt, sms, st, p);           \
            else launch_gs(k_grad<Tin, G_, false, true>, wt, sms, st, p);              \
        } else {                                                                       \
            if (vec) launch_gs(k_grad<Tin, G_, true, false>, wt, sms, st, p);          \
            else launch_gs(k_grad<Tin, G_, false, false>, wt, sms, st, p);             \
        }                                                                              \
    } while (0)
    if (V >= 512) GRADK(32);
    else if (V >= 128) GRADK(16);
    else if (V >= 32) GRADK(8);
    else GRADK(4);
#undef GRADK
    return true;
}

void* g_trace = nullptr;     // rnnt_set_trace: device buffer of int4 records
size_t g_trace_bytes = 0;

int g_coop[64];

bool coop_supported(int dev) {
    if (dev < 0 || dev >= 64) return false;
    if (!g_coop[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev);
        g_coop[dev] = v ? 1 : -1;
    }
    return g_coop[dev] > 0;
}

// Persistent path: every row, DP and gradient task in one cooperative launch.
// persistent_setup decides whether a call's shape is covered and, if so, the
// kernel, its shared memory and grid; launch_persistent then launches it.
struct PersistentCfg {
    const void* fn;
    size_t smem;
    int grid, zero_off, zero_rows, n_dp_sms;
};

template <typename Tin>
bool persistent_setup(const Params& p, int sms, int dev, PersistentCfg& c) {
    if (!coop_supported(dev)) return false;
    const char* env = getenv("RNNT_GB300_SCHEDULE");
    if (env && env[0] == 'k') return false;   // "kernels": one launch per stage
    constexpr int EPV = Elt<Tin>::kPerVec;
    const int V = p.V, nvec = V / EPV;
    const bool vec = ((size_t)V * sizeof(Tin)) % 16 == 0;
    // Its DP task runs lattices of at most two columns per lane (W <= 256).
    if (dp_jclass(dp_slots(p.S + 1)) > 2) return false;
    const size_t dps = dp_smem_for(p.S);
    const void* fn = nullptr;
    size_t sm = dps;
    int zero_off = 0, zero_rows = 0;
    // Log-softmax on short rows that are not 16-byte vectors (at most 1 KB):
    // plain loads, G-lane groups of plain_group(V) lanes per row.
    const bool plain = p.fused && !vec && (size_t)V * sizeof(Tin) <= 1024;
    if (p.fused && !plain) {
        if (!(vec && nvec > 32 && nvec <= 256)) return false;
        sm = std::max(sm, (size_t)8 * main_stages(nvec <= 64 ? 2 : nvec <= 128 ? 4 : 8) *
                              p.stage_bytes);
        sm = (sm + 127) / 128 * 128;
        const int rb = V * (int)sizeof(Tin);
        // Zero-row buffer from what is left of the dynamic shared memory that
        // still lets two CTAs share an SM (228 KB per SM, ~8.3 KB static and
        // 1 KB reserved per CTA).
        constexpr int kTwoCtaSmem = 104 * 1024;
        const int room = sm < kTwoCtaSmem ? (int)(kTwoCtaSmem - sm) / rb : 0;
        zero_rows = std::max(1, std::min(16384 / rb, room));
        zero_off = (int)sm;
        sm += (size_t)zero_rows * rb;
        fn = nvec <= 64    ? reinterpret_cast<const void*>(k_main<Tin, 2, 32, true>)
             : nvec <= 128 ? reinterpret_cast<const void*>(k_main<Tin, 4, 32, true>)
                           : reinterpret_cast<const void*>(k_main<Tin, 8, 32, true>);
    } else {
        if (flat_rows(V, sizeof(Tin), p.fused))   // shared staging of short rows
            sm = std::max(sm, (size_t)8 * flat_warp_bytes(V, sizeof(Tin)));
        const bool wide = plain ? plain_group(V) == 32 : V >= 256;
        fn = vec ? (wide ? reinterpret_cast<const void*>(k_main<Tin, 0, 32, true>)
                         : reinterpret_cast<const void*>(k_main<Tin, 0, 8, true>))
                 : (wide ? reinterpret_cast<const void*>(k_main<Tin, 0, 32, false>)
                         : reinterpret_cast<const void*>(k_main<Tin, 0, 8, false>));
    }
    if (sm > 110 * 1024) return false;
    const int occ = occupancy(fn, sm);
    if (occ < 1) return false;
    c.fn = fn;
    c.smem = sm;
    c.grid = occ * sms;
    c.zero_off = zero_off;
    c.zero_rows = zero_rows;
    // DP workers: up to 6 SMs (two DP CTAs each); measured on the BPE-ASR
    // workload, 6 beat 8 (the DP SMs idle most of the call) and 4.  A call of
    // short rows (under 64 MB of logits) is bound by its recursions, not by
    // HBM: there every sample's recursion gets a worker CTA, up to a quarter
    // of the SMs.
    const bool small = (double)p.rows * V * sizeof(Tin) < 64.0 * (1 << 20);
    c.n_dp_sms = small ? std::min((p.B + 1) / 2, sms / 4)
                       : std::min(std::min(6, (p.B + 1) / 2), sms / 8);
    return true;
}

// Returns false (nothing launched) when this shape is not covered or the
// cooperative launch is refused.
template <typename Tin>
bool launch_persistent(const Params& p, cudaStream_t st, int sms, int dev) {
    PersistentCfg c;
    if (!persistent_setup<Tin>(p, sms, dev, c)) return false;
    Params q = p;
    q.n_dp_sms = c.n_dp_sms;
    q.build_tasks = 1;
    q.zero_off = c.zero_off;
    q.zero_rows = c.zero_rows;
    void* args[] = {&q};
    if (cudaLaunchCooperativeKernel(c.fn, dim3(c.grid), dim3(256), args, c.smem, st) !=
        cudaSuccess) {
        cudaGetLastError();   // not launched: the caller runs the staged kernels instead
        return false;
    }
    return true;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

}  // namespace

extern "C" rnnt_status_t rnnt_workspace_size(int32_t B, int64_t rows, int32_t V, rnnt_dtype_t dt,
                                             size_t* bytes) {
    if (!bytes || B < 1 || rows < 1 || V < 1 || !valid_dtype(dt))
        return RNNT_INVALID_VALUE;
    *bytes = ws_total(B, rows, V, dt);
    return RNNT_OK;
}

// Every loss entry point: argument checks, then the persistent kernel or the
// staged kernels.  opts may be null (compact layout, no FastEmit).
static rnnt_status_t loss_impl(const void* logits, rnnt_dtype_t dt, int64_t rows, int32_t V,
                        const int32_t* targets, int32_t targets_stride,
                        const int32_t* logit_lengths, const int32_t* target_lengths, int32_t B,
                        int32_t blank, float clamp, int32_t fused_log_softmax,
                        rnnt_reduction_t reduction, float* loss, float* loss_reduced, void* grad,
                        void* workspace, size_t workspace_bytes, int32_t* status_dev,
                        rnnt_stream_t stream, const rnnt_options_t* opts,
                        void* const* stage_events) {
    if (!logits || !targets || !logit_lengths || !target_lengths || !loss || !workspace)
        return RNNT_INVALID_VALUE;
    float fe = 0.0f, sigma = 0.0f;
    int padded = 0, maxT = 0, maxW = 0, K = 0;
    int bb_id[RNNT_MAX_BIG_BLANKS] = {}, bb_dur[RNNT_MAX_BIG_BLANKS] = {};
    if (opts) {
        fe = opts->fastemit_lambda;
        if (!(fe >= 0.0f) || !(fe < INFINITY)) return RNNT_INVALID_VALUE;
        sigma = opts->sigma;
        if (!(sigma >= 0.0f) || !(sigma < INFINITY)) return RNNT_INVALID_VALUE;
        K = opts->num_big_blanks;
        if (K < 0 || K > RNNT_MAX_BIG_BLANKS) return RNNT_INVALID_VALUE;
        if (V < 1 || blank < -V || blank >= V) return RNNT_INVALID_VALUE;
        const int bl = blank < 0 ? blank + V : blank;
        for (int i = 0; i < K; ++i) {
            const int id = opts->big_blank_ids[i], dur = opts->big_blank_durations[i];
            if (id < -V || id >= V || dur < 2 || dur > RNNT_MAX_BIG_BLANK_DURATION)
                return RNNT_INVALID_VALUE;
            bb_id[i] = id < 0 ? id + V : id;
            bb_dur[i] = dur;
            if (bb_id[i] == bl) return RNNT_INVALID_VALUE;
            for (int j = 0; j < i; ++j)
                if (bb_id[j] == bb_id[i]) return RNNT_INVALID_VALUE;
        }
        if (opts->padded) {
            padded = 1;
            maxT = opts->max_T;
            maxW = opts->max_U + 1;
            if (maxT < 1 || opts->max_U < 0 || opts->max_U > RNNT_MAX_TARGET_LENGTH)
                return RNNT_INVALID_VALUE;
            if ((int64_t)maxT * maxW > INT32_MAX || B < 1 || rows != (int64_t)B * maxT * maxW)
                return RNNT_INVALID_VALUE;
        }
    }
    if (!valid_dtype(dt)) return RNNT_INVALID_VALUE;
    if (B < 1 || rows < 1 || V < 1 || rows < B) return RNNT_INVALID_VALUE;
    if (targets_stride < 1 || targets_stride > RNNT_MAX_TARGET_LENGTH) return RNNT_INVALID_VALUE;
    if (blank < -V || blank >= V) return RNNT_INVALID_VALUE;
    if (reduction != RNNT_RED_NONE && reduction != RNNT_RED_SUM && reduction != RNNT_RED_MEAN)
        return RNNT_INVALID_VALUE;
    if (!(clamp == clamp)) return RNNT_INVALID_VALUE;
    const size_t es = dt == RNNT_F32 ? 4 : 2;
    if (((uintptr_t)logits & 15) || (grad && ((uintptr_t)grad & 15)) || ((uintptr_t)workspace & 255))
        return RNNT_INVALID_VALUE;
    const size_t nbytes = (size_t)rows * (size_t)V * es;
    if (grad && grad != logits && overlaps(grad, nbytes, logits, nbytes)) return RNNT_INVALID_VALUE;
    const Layout L = ws_layout(B, rows);
    const bool multiblank = K > 0 || sigma > 0.0f;
    if (workspace_bytes < (multiblank ? ws_total_mb(B, rows, K) : ws_total(B, rows, V, dt)))
        return RNNT_WORKSPACE_TOO_SMALL;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RNNT_LAUNCH_FAILED;
    const int sms = num_sms(dev);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    char* w = static_cast<char*>(workspace);
    Params p{};
    p.logits = logits;
    p.grad = grad;
    p.rows = rows;
    p.V = V;
    p.dt = dt;
    p.targets = targets;
    p.S = targets_stride;
    p.Tl = logit_lengths;
    p.Ul = target_lengths;
    p.B = B;
    p.blank = blank < 0 ? blank + V : blank;
    p.clamp = clamp > 0.0f ? clamp : INFINITY;
    p.scale = reduction == RNNT_RED_MEAN ? 1.0f / (float)B : 1.0f;
    // A row whose occupancy is below 2^skip2 has every |grad| below half the
    // smallest subnormal of the output type, so every element rounds to zero.
    // (Smallest subnormals: 2^-24 fp16, 2^-133 bf16, 2^-149 fp32.)
    const float zero_at = dt == RNNT_F16 ? -25.5f : (dt == RNNT_BF16 ? -134.5f : -151.0f);
    p.skip2 = zero_at - log2f(p.scale);
    p.lscale = log2f(p.scale);
    p.fused = fused_log_softmax ? 1 : 0;
    p.red = reduction;
    p.fe = fe;
    p.fe_l2 = log2f(1.0f + fe);
    p.padded = padded;
    p.maxT = maxT;
    p.maxW = maxW;
    p.K = K;
    for (int i = 0; i < RNNT_MAX_BIG_BLANKS; ++i) {
        p.bb_id[i] = bb_id[i];
        p.bb_dur[i] = bb_dur[i];
    }
    p.bb_c = (float)exp(-(double)sigma);
    p.pbb = multiblank ? reinterpret_cast<int2*>(static_cast<char*>(workspace) + L.total) : nullptr;
    p.stage_bytes = (int)(((size_t)V * es + 127) / 128 * 128);
    p.loss = loss;
    p.loss_red = loss_reduced;
    p.status = status_dev;
    p.err = reinterpret_cast<int32_t*>(w + L.err);
    p.off = reinterpret_cast<int64_t*>(w + L.off);
    p.order = reinterpret_cast<int32_t*>(w + L.order);
    p.lossa = reinterpret_cast<double*>(w + L.lossa);
    p.lossb = reinterpret_cast<double*>(w + L.lossb);
    p.pm = reinterpret_cast<float*>(w + L.pm);
    p.pe = reinterpret_cast<int32_t*>(w + L.pe);
    p.lse2 = reinterpret_cast<float*>(w + L.lse2);
    p.info = (!multiblank && long_rows(V, dt)) ? reinterpret_cast<float4*>(w + L.total) : nullptr;
    p.edge = reinterpret_cast<int4*>(w + L.edge);
    p.alpha = reinterpret_cast<int2*>(w + L.alpha);
    p.beta = reinterpret_cast<int2*>(w + L.beta);
    p.rtasks = reinterpret_cast<int32_t*>(w + L.rtasks);
    p.rdone = reinterpret_cast<int32_t*>(w + L.rdone);
    p.dpdone = reinterpret_cast<int32_t*>(w + L.dpdone);
    p.dpclaim = reinterpret_cast<int32_t*>(w + L.dpclaim);
    p.tasks = reinterpret_cast<int4*>(w + L.tasks);
    p.trace = static_cast<int4*>(g_trace);
    p.trace_cap = (int64_t)(g_trace_bytes / sizeof(int4));

    const size_t dp_smem = dp_smem_dir_for(targets_stride);
    if (dev >= 0 && dev < 64 && g_dp_smem_set[dev] < (int)dp_smem) {
        if (cudaFuncSetAttribute(k_dp, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dp_smem) !=
            cudaSuccess)
            return RNNT_LAUNCH_FAILED;
        g_dp_smem_set[dev] = (int)dp_smem;
    }

    auto mark = [&](int i) {
        if (stage_events && stage_events[i])
            cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), st);
    };
    // Without the in-kernel log-softmax (single blank, per-stage kernels) the
    // recursion launch also zeroes the whole gradient buffer, padding rows
    // included, and the gradient pass writes only the blank and label
    // elements.  (The persistent kernel, when it takes the call, writes every
    // row itself.)
    const bool persistent_shape = grad && !multiblank && with_type(dt, [&](auto tag) {
        PersistentCfg c;
        return persistent_setup<decltype(tag)>(p, sms, dev, c);
    });
    const bool sparse = grad && !multiblank && !fused_log_softmax && !persistent_shape;
    mark(0);
    if (grad && padded && !sparse) {   // zero gradient rows outside the lattices
        with_type(dt, [&](auto tag) {
            launch_gs(k_pad_zero<decltype(tag)>, rows * 32, sms, st, p);
            return 0;
        });
    }
    if (multiblank) {
        // Multi-blank transducer: preparation, the row pass (also storing every
        // big blank's probability), the recursions, the gradient rows, the check.
        const int nthr = std::min(1024, (targets_stride + 1 + 31) / 32 * 32);
        const size_t smem = (size_t)(kMbRing + 2) * nthr * sizeof(float2) +
                            (size_t)kMbRing * nthr * sizeof(int);
        const void* kmb = nthr <= 256 ? reinterpret_cast<const void*>(k_dp_mb<256>)
                                      : reinterpret_cast<const void*>(k_dp_mb<1024>);
        if (cudaFuncSetAttribute(kmb, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return RNNT_LAUNCH_FAILED;
        k_prepare<<<1, 1024, 0, st>>>(p);
        with_type(dt, [&](auto tag) {
            launch_rows<decltype(tag)>(p, st, sms);
            return 0;
        });
        if (nthr <= 256) k_dp_mb<256><<<dim3(B, 2), nthr, smem, st>>>(p);
        else k_dp_mb<1024><<<dim3(B, 2), nthr, smem, st>>>(p);
        bool finalized = false;
        if (grad) {
            finalized = with_type(dt, [&](auto tag) {
                using T = decltype(tag);
                const int nv = V / Elt<T>::kPerVec;
                if (fused_log_softmax && ((size_t)V * sizeof(T)) % 16 == 0 && nv > 32 &&
                    nv <= 256) {
                    // Rows staged by TMA (as the standard gradient pass); its last
                    // CTA runs the loss check.
                    const size_t sm = tma_smem(p);
                    const int64_t wt = (rows + 31) / 32 * 32;
                    if (nv <= 64) launch_gs(k_grad_tma<T, 2, true>, wt, sms, st, p, sm);
                    else if (nv <= 128) launch_gs(k_grad_tma<T, 4, true>, wt, sms, st, p, sm);
                    else launch_gs(k_grad_tma<T, 8, true>, wt, sms, st, p, sm);
                    return true;
                }
                if (((size_t)V * sizeof(T)) % 16 == 0)
                    launch_gs(k_grad_mb<T, true>, rows * 32, sms, st, p);
                else
                    launch_gs(k_grad_mb<T, false>, rows * 32, sms, st, p);
                return false;
            });
        }
        if (!finalized) k_finalize<<<1, 256, 0, st>>>(p);
        for (int i = 1; i <= 6; ++i) mark(i);
        return cudaGetLastError() == cudaSuccess ? RNNT_OK : RNNT_LAUNCH_FAILED;
    }
    if (grad) {
        // One cooperative kernel: preparation on its CTA 0, every task, and the
        // loss check / reduction on its last CTA.
        const bool done = with_type(
            dt, [&](auto tag) { return launch_persistent<decltype(tag)>(p, st, sms, dev); });
        if (done) {
            for (int i = 1; i <= 6; ++i) mark(i);
            return cudaGetLastError() == cudaSuccess ? RNNT_OK : RNNT_LAUNCH_FAILED;
        }
    }
    k_prepare<<<1, 1024, 0, st>>>(p);
    mark(1);
    with_type(dt, [&](auto tag) {
        launch_rows<decltype(tag)>(p, st, sms);
        return 0;
    });
    mark(2);
    int zy = 0;   // rows of zero-fill CTAs in the recursion launch's grid
    if (sparse) {
        p.zfill = (int64_t)nbytes;
        p.zcta = sms;
        p.zbuf = (int)(std::min(dp_smem, (size_t)32768) & ~size_t(15));
        p.info = nullptr;
        zy = (sms + B - 1) / B;
    }
    k_dp<<<dim3(B, 2 + zy), dp_threads_for(targets_stride), dp_smem, st>>>(p);
    mark(3);
    if (grad && p.info) launch_gs(k_combine, rows, sms, st, p);   // long rows: the records first
    mark(4);   // (otherwise the gradient records are formed inside the gradient kernel)
    if (grad) {
        // The gradient kernel's last CTA also runs the loss check / reduction
        // (except the long-row kernel's: a check kernel follows it).
        const bool checked = with_type(dt, [&](auto tag) {
            using T = decltype(tag);
            if (sparse) {
                k_grad_sparse<T><<<(unsigned)((rows + kSparseRows - 1) / kSparseRows), 256, 0, st>>>(p);
                return true;
            }
            return launch_grad<T>(p, st, sms);
        });
        mark(5);
        if (!checked) k_finalize<<<1, 256, 0, st>>>(p);
    } else {
        mark(5);
        k_finalize<<<1, 256, 0, st>>>(p);
    }
    mark(6);
    return cudaGetLastError() == cudaSuccess ? RNNT_OK : RNNT_LAUNCH_FAILED;
}

extern "C" rnnt_status_t rnnt_workspace_size_ex(int32_t B, int64_t rows, int32_t V,
                                                rnnt_dtype_t dt, const rnnt_options_t* options,
                                                size_t* bytes) {
    if (!bytes || B < 1 || rows < 1 || V < 1 || !valid_dtype(dt)) return RNNT_INVALID_VALUE;
    const int K = options ? options->num_big_blanks : 0;
    if (K < 0 || K > RNNT_MAX_BIG_BLANKS) return RNNT_INVALID_VALUE;
    const bool mb = options && (K > 0 || options->sigma > 0.0f);
    *bytes = mb ? ws_total_mb(B, rows, K) : ws_total(B, rows, V, dt);
    return RNNT_OK;
}

extern "C" rnnt_status_t rnnt_loss_fused_staged(
    const void* logits, rnnt_dtype_t dt, int64_t rows, int32_t V, const int32_t* targets,
    int32_t targets_stride, const int32_t* logit_lengths, const int32_t* target_lengths, int32_t B,
    int32_t blank, float clamp, int32_t fused_log_softmax, rnnt_reduction_t reduction, float* loss,
    float* loss_reduced, void* grad, void* workspace, size_t workspace_bytes, int32_t* status_dev,
    rnnt_stream_t stream, void* const* stage_events) {
    return loss_impl(logits, dt, rows, V, targets, targets_stride, logit_lengths, target_lengths,
                     B, blank, clamp, fused_log_softmax, reduction, loss, loss_reduced, grad,
                     workspace, workspace_bytes, status_dev, stream, nullptr, stage_events);
}

extern "C" rnnt_status_t rnnt_loss_fused_ex(
    const void* logits, rnnt_dtype_t dt, int64_t rows, int32_t V, const int32_t* targets,
    int32_t targets_stride, const int32_t* logit_lengths, const int32_t* target_lengths, int32_t B,
    int32_t blank, float clamp, int32_t fused_log_softmax, rnnt_reduction_t reduction, float* loss,
    float* loss_reduced, void* grad, void* workspace, size_t workspace_bytes, int32_t* status_dev,
    rnnt_stream_t stream, const rnnt_options_t* options) {
    return loss_impl(logits, dt, rows, V, targets, targets_stride, logit_lengths, target_lengths,
                     B, blank, clamp, fused_log_softmax, reduction, loss, loss_reduced, grad,
                     workspace, workspace_bytes, status_dev, stream, options, nullptr);
}

extern "C" rnnt_status_t rnnt_loss_fused(const void* logits, rnnt_dtype_t dt, int64_t rows, int32_t V,
                                         const int32_t* targets, int32_t targets_stride,
                                         const int32_t* logit_lengths, const int32_t* target_lengths,
                                         int32_t B, int32_t blank, float clamp,
                                         int32_t fused_log_softmax, rnnt_reduction_t reduction,
                                         float* loss, float* loss_reduced, void* grad,
                                         void* workspace, size_t workspace_bytes,
                                         int32_t* status_dev, rnnt_stream_t stream) {
    return rnnt_loss_fused_staged(logits, dt, rows, V, targets, targets_stride, logit_lengths,
                                  target_lengths, B, blank, clamp, fused_log_softmax, reduction,
                                  loss, loss_reduced, grad, workspace, workspace_bytes, status_dev,
                                  stream, nullptr);
}

extern "C" rnnt_status_t rnnt_grad_scale(void* grad, rnnt_dtype_t dt, int64_t rows, int32_t V,
                                         int32_t B, const void* workspace, size_t workspace_bytes,
                                         const float* factors, int32_t per_sample,
                                         rnnt_stream_t stream) {
    if (!grad || !workspace || !factors || rows < 1 || V < 1 || B < 1) return RNNT_INVALID_VALUE;
    if (!valid_dtype(dt)) return RNNT_INVALID_VALUE;
    const Layout L = ws_layout(B, rows);
    if (workspace_bytes < L.total) return RNNT_WORKSPACE_TOO_SMALL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RNNT_LAUNCH_FAILED;
    const int grid = grid_for(rows * 32, num_sms(dev), 4);
    const char* w = static_cast<const char*>(workspace);
    const int64_t* off = reinterpret_cast<const int64_t*>(w + L.off);
    const int32_t* hdr = reinterpret_cast<const int32_t*>(w + L.err);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    with_type(dt, [&](auto tag) {
        k_scale<decltype(tag)><<<grid, 256, 0, st>>>(grad, rows, V, B, off, hdr, factors,
                                                     per_sample);
        return 0;
    });
    return cudaGetLastError() == cudaSuccess ? RNNT_OK : RNNT_LAUNCH_FAILED;
}

extern "C" rnnt_status_t rnnt_plan(int32_t B, int64_t rows, int32_t V, rnnt_dtype_t dt,
                                   int32_t targets_stride, int32_t fused_log_softmax,
                                   int32_t want_grad, const rnnt_options_t* options,
                                   rnnt_plan_t* plan) {
    if (!plan || B < 1 || rows < 1 || V < 1 || !valid_dtype(dt)) return RNNT_INVALID_VALUE;
    if (targets_stride < 1 || targets_stride > RNNT_MAX_TARGET_LENGTH) return RNNT_INVALID_VALUE;
    const int K = options ? options->num_big_blanks : 0;
    if (K < 0 || K > RNNT_MAX_BIG_BLANKS) return RNNT_INVALID_VALUE;
    const bool multiblank = options && (K > 0 || options->sigma > 0.0f);
    const int pad = (options && options->padded && want_grad) ? 1 : 0;
    const int g = want_grad ? 1 : 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RNNT_LAUNCH_FAILED;
    }
    plan->persistent = 0;
    if (multiblank) {   // prepare, rows, recursions, gradient rows, check
        // (the TMA-staged gradient kernel, for log-softmax on rows of 33 to 256
        // 16-byte vectors, runs the check itself)
        const int epv = dt == RNNT_F32 ? 4 : 8;
        const int nv = V / epv;
        const bool tma = want_grad && fused_log_softmax && V % epv == 0 && nv > 32 && nv <= 256;
        plan->launches = pad + 4 + g - (tma ? 1 : 0);
        return RNNT_OK;
    }
    if (want_grad) {
        Params p{};
        p.B = B;
        p.V = V;
        p.S = targets_stride;
        p.fused = fused_log_softmax ? 1 : 0;
        const size_t es = dt == RNNT_F32 ? 4 : 2;
        p.stage_bytes = (int)(((size_t)V * es + 127) / 128 * 128);
        PersistentCfg c;
        const bool ok = with_type(dt, [&](auto tag) {
            return persistent_setup<decltype(tag)>(p, num_sms(dev), dev, c);
        });
        if (ok) {
            plan->persistent = 1;
            plan->launches = pad + 1;
            return RNNT_OK;
        }
    }
    // prepare, rows, recursions, [long rows: records], gradient, [long rows: check];
    // without the log-softmax: prepare, rows, recursions (and zero-fill), the
    // blank / label elements (and check)
    if (want_grad && !fused_log_softmax) plan->launches = 4;
    else plan->launches = pad + 4 + ((want_grad && long_rows(V, dt)) ? 2 : 0);
    return RNNT_OK;
}

extern "C" rnnt_status_t rnnt_selftest_wait_timeout(int32_t* status_dev, int32_t polls,
                                                    rnnt_stream_t stream) {
    if (!status_dev || polls < 1) return RNNT_INVALID_VALUE;
    k_selftest_wait<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status_dev, polls);
    return cudaGetLastError() == cudaSuccess ? RNNT_OK : RNNT_LAUNCH_FAILED;
}

extern "C" rnnt_status_t rnnt_set_trace(void* device_buffer, size_t bytes) {
    if (device_buffer && ((uintptr_t)device_buffer & 15)) return RNNT_INVALID_VALUE;
    g_trace = bytes >= sizeof(int4) ? device_buffer : nullptr;
    g_trace_bytes = g_trace ? bytes : 0;
    return RNNT_OK;
}

extern "C" const char* rnnt_status_string(rnnt_status_t s) {
    switch (s) {
        case RNNT_OK: return "success";
        case RNNT_INVALID_VALUE: return "invalid value (arguments, lengths or targets)";
        case RNNT_WORKSPACE_TOO_SMALL: return "workspace too small";
        case RNNT_LAUNCH_FAILED: return "kernel launch failed";
        case RNNT_LOSS_MISMATCH: return "alpha/beta loss mismatch or non-finite input";
        case RNNT_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

extern "C" int32_t rnnt_abi_version(void) { return 103; }

// ---------------------------------------------------------------- no-alloc entry
// rnnt_loss_fused_noalloc runs rnnt_loss_fused over a fixed scratch array of
// this module instead of a caller workspace.  The array's device address is
// looked up once per device (with that device current) and cached; the
// lookup allocates nothing.  The workspace path rewrites every scratch word
// it reads (k_prepare resets the counters, offsets and task list first), so
// the contents a previous call left need no clearing.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[RNNT_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoallocMaxDevices] = {};

}  // namespace

extern "C" rnnt_status_t rnnt_loss_fused_noalloc(
    const void* logits, rnnt_dtype_t dt, int64_t rows, int32_t V, const int32_t* targets,
    int32_t targets_stride, const int32_t* logit_lengths, const int32_t* target_lengths, int32_t B,
    int32_t blank, float clamp, int32_t fused_log_softmax, rnnt_reduction_t reduction, float* loss,
    float* loss_reduced, void* grad, int32_t* status_dev, rnnt_stream_t stream) {
    if (B < 1 || rows < 1 || V < 1 || !valid_dtype(dt)) return RNNT_INVALID_VALUE;
    const size_t need = ws_total(B, rows, V, dt);
    if (need > RNNT_NOALLOC_SCRATCH_BYTES) return RNNT_WORKSPACE_TOO_SMALL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices)
        return RNNT_LAUNCH_FAILED;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        if (!g_noalloc_ptr[dev]) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
                cudaGetLastError();   // leave no error behind for the next launch check
                return RNNT_LAUNCH_FAILED;
            }
            g_noalloc_ptr[dev] = ptr;
        }
        scratch = g_noalloc_ptr[dev];
    }
    return rnnt_loss_fused(logits, dt, rows, V, targets, targets_stride, logit_lengths,
                           target_lengths, B, blank, clamp, fused_log_softmax, reduction, loss,
                           loss_reduced, grad, scratch, RNNT_NOALLOC_SCRATCH_BYTES, status_dev,
                           stream);
}
