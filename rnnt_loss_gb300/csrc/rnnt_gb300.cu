// rnnt_gb300.cu -- fused RNN-T loss forward+backward for GB300 (sm_103a).
//
// Device pipeline of one rnnt_loss_fused call (all on the caller's stream):
//   k_prepare   1 CTA: validates lengths/targets, exclusive int64 scan of
//               T_b*(U_b+1) (row offsets), largest-lattice-first sample order.
//               Replaces the host-side largest-task-first balancer of the
//               rnnt-loss-ascend README (架构设计 "Host 侧").
//   k_row_*     one pass over the logits: per row the log-softmax denominator
//               (single-pass max/sum, warp-shuffle reduction) and the blank /
//               target log-probs, scattered into an anti-diagonal-packed
//               layout for the DP (README 对角线遍历 α/β).  With the in-kernel
//               log-softmax off only the two needed elements are read.
//   k_dp        one CTA of two warps per sample: warp 0 runs the alpha
//               recursion over anti-diagonals d = 0..T+U-1, warp 1 the beta
//               recursion from the end; they meet at the middle diagonal,
//               swap frame offsets, and each then finishes its sweep while
//               combining alpha and beta of the half the other warp computed
//               into per-row gradient coefficients (README 核心梯度融合公式).
//   k_grad_*    one read + one write of the logits: grad_k =
//               p_k*occ - [k=blank]*post_blank - [k=y]*post_label, clip,
//               reduction scale, store in the input dtype (may alias logits).
//               Rows whose occupancy is too small to change any output value
//               are written as zeros without reading the logits.
//   k_finalize  1 CTA: alpha/beta loss cross-check (README 精度保证 "双 loss
//               互校验"), deterministic reduction, status word.
//
// Numerics: log-domain, base 2.  The DP keeps each anti-diagonal in a frame
// with an integer offset (a power-of-two scale in the probability domain), so
// fp32 values stay O(10) while the exact frame offsets carry the magnitude
// of the accumulated log-probability.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "rnnt_gb300.h"

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr double kLn2 = 0.69314718055994530942;
constexpr int kMaxW = RNNT_MAX_TARGET_LENGTH + 1;

enum : int {
    ERR_LENGTH = 1,
    ERR_ROWS = 2,
    ERR_TARGET = 4,
    ERR_MISMATCH = 8,
};

// ---------------------------------------------------------------- workspace
struct Layout {
    size_t err, off, order, lossa, lossb, delta, lse2, lpb, lpy, va, vb, oa, qb, info, total;
};

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
    L.delta = p; p = al256(p + sizeof(float) * (size_t)B);
    L.lse2 = p;  p = al256(p + sizeof(float) * R);
    L.lpb = p;   p = al256(p + sizeof(float) * R);
    L.lpy = p;   p = al256(p + sizeof(float) * R);
    L.va = p;    p = al256(p + sizeof(float) * R);
    L.vb = p;    p = al256(p + sizeof(float) * R);
    L.oa = p;    p = al256(p + sizeof(int32_t) * R);
    L.qb = p;    p = al256(p + sizeof(int32_t) * R);
    L.info = p;  p = al256(p + sizeof(float4) * R);
    L.total = p;
    return L;
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
    int fused;
    int red;
    int want_grad;
    int ring_floats;  // per-warp DP ring size (floats)
    float* loss;
    float* loss_red;
    int32_t* status;
    // workspace views
    int32_t* err;
    int64_t* off;
    int32_t* order;
    double* lossa;
    double* lossb;
    float* delta;
    float* lse2;
    float* lpb;
    float* lpy;
    float* va;
    float* vb;
    int32_t* oa;
    int32_t* qb;
    float4* info;
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
// log2(2^a + 2^b); -inf absorbing, NaN-free when both are -inf.
__device__ __forceinline__ float lae2(float a, float b) {
    float mx = fmaxf(a, b), mn = fminf(a, b);
    float dd = fmaxf(mn - mx, -126.0f);
    return mx + lg2(1.0f + ex2(dd));
}

// Number of lattice nodes (t,u), 0<=t<T, 0<=u<W, with t+u < d: first packed
// index of anti-diagonal d (inclusion-exclusion over the rectangle).
__device__ __forceinline__ int64_t tri(int64_t n) { return n > 0 ? n * (n + 1) / 2 : 0; }
__device__ __forceinline__ int64_t diag_start(int d, int T, int W) {
    return tri(d) - tri((int64_t)d - T) - tri((int64_t)d - W) + tri((int64_t)d - T - W);
}

__device__ __forceinline__ int find_sample(const int64_t* off, int B, int64_t r) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(off + mid) <= r) lo = mid; else hi = mid;
    }
    return lo;
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

// ---------------------------------------------------------------- k_prepare
__global__ void __launch_bounds__(1024) k_prepare(Params p) {
    __shared__ int64_t wsum[32];
    __shared__ int64_t carry;
    __shared__ int errs;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) { carry = 0; errs = 0; }
    __syncthreads();
    for (int base = 0; base < p.B; base += blockDim.x) {
        const int b = base + tid;
        int64_t n = 0;
        if (b < p.B) {
            const int T = p.Tl[b], U = p.Ul[b];
            if (T < 1 || U < 0 || U > p.S || U + 1 > kMaxW) atomicOr(&errs, ERR_LENGTH);
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
        if (carry != p.rows) atomicOr(&errs, ERR_ROWS);
    }
    // Labels: in range, not blank (warp-transducer blog 5.2).
    const int64_t nt = (int64_t)p.B * p.S;
    for (int64_t i = tid; i < nt; i += blockDim.x) {
        const int b = (int)(i / p.S), u = (int)(i % p.S);
        const int U = p.Ul[b];
        if (U >= 0 && U <= p.S && u < U) {
            const int y = p.targets[i];
            if (y < 0 || y >= p.V || y == p.blank) atomicOr(&errs, ERR_TARGET);
        }
    }
    // Largest DP first: key (T+U, area), ties by index.  O(B^2) rank sort.
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
    if (tid == 0) *p.err = errs;
}

// ---------------------------------------------------------------- row pass
// Writes, at the packed index of node (t,u):
//   lse2 = log2 sum_k 2^(h_k log2e)     (0 with the in-kernel softmax off)
//   lpb  = log2 P(blank|t,u), -inf at t=T-1, u<U (no blank leaves the last frame
//          before every label is out)
//   lpy  = log2 P(y_{u+1}|t,u), -inf at u=U
__device__ __forceinline__ void row_store(const Params& p, int b, int64_t r, float lse2v,
                                          float hb, float hy) {
    const int T = __ldg(p.Tl + b), U = __ldg(p.Ul + b), W = U + 1;
    const int64_t o = __ldg(p.off + b);
    const int64_t rr = r - o;
    const int t = (int)(rr / W), u = (int)(rr - (int64_t)t * W);
    const int d = t + u;
    const int64_t idx = o + diag_start(d, T, W) + (t - max(0, d - U));
    p.lse2[idx] = lse2v;
    p.lpb[idx] = (t == T - 1 && u < U) ? -INFINITY : hb * kLog2e - lse2v;
    p.lpy[idx] = (u < U) ? hy * kLog2e - lse2v : -INFINITY;
}

__device__ __forceinline__ int row_label(const Params& p, int b, int64_t r) {
    const int U = __ldg(p.Ul + b), W = U + 1;
    const int64_t rr = r - __ldg(p.off + b);
    const int u = (int)(rr % W);
    return (u < U) ? __ldg(p.targets + (int64_t)b * p.S + u) : -1;
}

template <typename Tin, int G, bool VEC>
__global__ void __launch_bounds__(256) k_row_fused(Params p) {
    if (*p.err) return;
    using E = Elt<Tin>;
    const Tin* X = static_cast<const Tin*>(p.logits);
    const int V = p.V;
    const int lane = threadIdx.x & (G - 1);
    const unsigned gm = group_mask<G>();
    const int64_t ng = (int64_t)gridDim.x * (blockDim.x / G);
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / G; r < p.rows; r += ng) {
        const Tin* row = X + r * (int64_t)V;
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
                }
            }
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) {
            const float om = __shfl_xor_sync(gm, m, o, G);
            const float os = __shfl_xor_sync(gm, s, o, G);
            const float nm = fmaxf(m, om);
            if (nm != -INFINITY) s = s * ex2((m - nm) * kLog2e) + os * ex2((om - nm) * kLog2e);
            m = nm;
        }
        if (lane == 0) {
            const float lse2v = m * kLog2e + lg2(s);
            const int b = find_sample(p.off, p.B, r);
            const int y = row_label(p, b, r);
            const float hb = E::get(row, p.blank);
            const float hy = (y >= 0) ? E::get(row, y) : 0.0f;
            row_store(p, b, r, lse2v, hb, hy);
        }
    }
}

// In-kernel log-softmax off: the rows already hold log-probs; read 2 elements.
template <typename Tin>
__global__ void __launch_bounds__(256) k_row_gather(Params p) {
    if (*p.err) return;
    using E = Elt<Tin>;
    const Tin* X = static_cast<const Tin*>(p.logits);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < p.rows; r += stride) {
        const Tin* row = X + r * (int64_t)p.V;
        const int b = find_sample(p.off, p.B, r);
        const int y = row_label(p, b, r);
        const float hb = E::get(row, p.blank);
        const float hy = (y >= 0) ? E::get(row, y) : 0.0f;
        row_store(p, b, r, 0.0f, hb, hy);
    }
}

// ---------------------------------------------------------------- DP
// Per-warp ring of prefetched anti-diagonal data in shared memory.  Slot
// layout (floats): [lpb J*32][lpy J*32][lse2 J*32][v_other J*32][frame 32];
// column u = lane + 32*j.  Ring depth R, prefetch distance R-2.
template <int J> struct Ring;
template <> struct Ring<1> { static constexpr int R = 32; };
template <> struct Ring<2> { static constexpr int R = 32; };
template <> struct Ring<4> { static constexpr int R = 16; };
template <> struct Ring<8> { static constexpr int R = 8; };
template <> struct Ring<16> { static constexpr int R = 6; };
template <> struct Ring<32> { static constexpr int R = 4; };

__host__ __device__ constexpr int ring_slot_floats(int J) { return (4 * J + 1) * 32; }

__device__ __forceinline__ void cp4(void* smem, const void* gmem) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }
__device__ __forceinline__ void cp_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

struct Samp {
    int b, T, U, W, D, dm;
    int64_t off;
};

// Queue the loads of anti-diagonal d into its ring slot: edge log-weights
// always, and (when `comb`) lse2, the other direction's values and frame.
template <int J>
__device__ __forceinline__ void ring_issue(const Samp& c, float* ring, int d, bool comb,
                                           const float* lpb, const float* lpy, const float* lse2,
                                           const float* vo, const int32_t* fo, int lane) {
    constexpr int R = Ring<J>::R, SL = ring_slot_floats(J);
    if (d >= 0 && d < c.D) {
        float* sl = ring + (d % R) * SL;
        const int64_t base = c.off + diag_start(d, c.T, c.W) - max(0, d - c.U) + d;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int u = lane + 32 * j, t = d - u;
            float* e = sl + j * 32 + lane;
            if (u <= c.U && t >= 0 && t < c.T) {
                const int64_t g = base - u;
                cp4(e, lpb + g);
                cp4(e + J * 32, lpy + g);
                if (comb) {
                    cp4(e + 2 * J * 32, lse2 + g);
                    cp4(e + 3 * J * 32, vo + g);
                }
            } else {
                e[0] = -INFINITY;
                e[J * 32] = -INFINITY;
                if (comb) {
                    e[2 * J * 32] = 0.0f;
                    e[3 * J * 32] = -INFINITY;
                }
            }
        }
        if (comb) cp4(sl + 4 * J * 32 + lane, fo + c.off + d);
    }
}

template <int J>
__device__ __forceinline__ float warp_max_valid(const float* v, int d, const Samp& c, int lane) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < J; ++j) {
        const int u = lane + 32 * j, t = d - u;
        if (u <= c.U && t >= 0 && t < c.T) m = fmaxf(m, v[j]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    return m;
}

// Gradient coefficients of node (t,u) on anti-diagonal e (all log2, relative
// to the sample's reference frame C; the per-sample correction C - ll is
// added by the gradient pass):
//   x: log2(occupancy) - lse2    y: log2(occupancy)
//   z: log2(posterior of the blank arc)   w: log2(posterior of the label arc)
__device__ __forceinline__ void put_info(const Params& p, const Samp& c, int t, int u, float va,
                                         float vbe, float lpb, float lpy, float lse2v,
                                         float vb_blank, float vb_label, float KA, float KB) {
    const float lc = va + vbe + KA;
    float eb;
    if (t < c.T - 1) eb = va + lpb + vb_blank + KB;
    else eb = (u == c.U) ? lc : -INFINITY;
    const float ey = (u < c.U) ? va + lpy + vb_label + KB : -INFINITY;
    p.info[c.off + (int64_t)t * c.W + u] = make_float4(lc - lse2v, lc, eb, ey);
}

template <int J>
__device__ void dp_alpha(const Params& p, const Samp& c, float* ring, int* xch) {
    constexpr int R = Ring<J>::R, PF = R - 2, SL = ring_slot_floats(J);
    const int lane = threadIdx.x & 31;
    float v[J];
#pragma unroll
    for (int j = 0; j < J; ++j) v[j] = (lane + 32 * j == 0) ? 0.0f : -INFINITY;
    if (lane == 0) {
        p.va[c.off] = 0.0f;
        p.oa[c.off] = 0;
    }
    for (int k = 0; k <= PF; ++k) {
        ring_issue<J>(c, ring, k, false, p.lpb, p.lpy, p.lse2, p.vb, p.qb, lane);
        cp_commit();
    }
    // Integer frame offsets (log2 units) of diagonals d-1..d-4 and the warp
    // maxima of v on d-2..d-4 (each in its own frame).  The frame of d is
    // extrapolated from the maxima of d-3 and d-4, whose reductions have two
    // iterations to complete, so they stay off the recursion's critical path.
    int O = 0, Oh2 = 0, Oh3 = 0, Oh4 = 0;
    float mA = -INFINITY, mB = -INFINITY, mC = -INFINITY;
    bool synced = false;
    int C = 0;
    const bool comb_on = p.want_grad != 0;

    for (int d = 1; d <= c.D; ++d) {
        if (d == c.dm + 1) {
            // Midpoint: swap frame offsets, then fetch what the combine needs.
            if (lane == 0) xch[0] = O;
            asm volatile("bar.sync 1, 64;\n" ::: "memory");
            C = xch[0] + xch[1];
            synced = true;
            if (comb_on) {
                for (int e = c.dm + 1; e <= min(c.dm + PF, c.D - 1); ++e) {
                    float* sl = ring + (e % R) * SL;
                    const int64_t base = c.off + diag_start(e, c.T, c.W) - max(0, e - c.U) + e;
#pragma unroll
                    for (int j = 0; j < J; ++j) {
                        const int u = lane + 32 * j, t = e - u;
                        float* q = sl + j * 32 + lane;
                        if (u <= c.U && t >= 0 && t < c.T) {
                            cp4(q + 2 * J * 32, p.lse2 + base - u);
                            cp4(q + 3 * J * 32, p.vb + base - u);
                        } else {
                            q[2 * J * 32] = 0.0f;
                            q[3 * J * 32] = -INFINITY;
                        }
                    }
                    cp4(sl + 4 * J * 32 + lane, p.qb + c.off + e);
                }
                cp_commit();
                cp_wait_all();
            }
        }
        if (d == c.D) break;
        ring_issue<J>(c, ring, d + PF, synced && comb_on, p.lpb, p.lpy, p.lse2, p.vb, p.qb, lane);
        cp_commit();
        cp_wait<PF>();
        __syncwarp();
        const float* sp = ring + ((d - 1) % R) * SL;
        const float* sc = ring + (d % R) * SL;

        int Onew = O;
        if (fabsf(mB) < 1e6f && fabsf(mC) < 1e6f) {
            const int a3 = Oh3 + (int)rintf(mB), a4 = Oh4 + (int)rintf(mC);
            Onew = a3 + 3 * (a3 - a4);
        }
        const int sig = Onew - O;
        const float sh = (float)sig;
        float ob[J], oy[J], yy[J], nv[J];
#pragma unroll
        for (int j = 0; j < J; ++j) {
            ob[j] = v[j] + (sp[j * 32 + lane] - sh);
            oy[j] = v[j] + (sp[(J + j) * 32 + lane] - sh);
        }
#pragma unroll
        for (int j = 0; j < J; ++j) yy[j] = __shfl_sync(0xffffffffu, oy[j], (lane + 31) & 31);
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const float nb = lane ? yy[j] : (j ? yy[j - 1] : -INFINITY);
            nv[j] = lae2(ob[j], nb);
        }
        // Lagged frame choice: the max of diagonal d-1 drives the shift at d+1.
        const float m_prev = warp_max_valid<J>(v, d - 1, c, lane);

        if (synced && comb_on && d - 1 > c.dm) {
            const int e = d - 1;
            const int Qe = __float_as_int(sp[4 * J * 32 + lane]);
            const int Qn = __float_as_int(sc[4 * J * 32 + lane]);
            const float KA = (float)(O + Qe - C), KB = (float)(O + Qn - C);
            float nbv[J];
#pragma unroll
            for (int j = 0; j < J; ++j)
                nbv[j] = __shfl_sync(0xffffffffu, sc[(3 * J + j) * 32 + lane], (lane + 1) & 31);
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int u = lane + 32 * j, t = e - u;
                if (u <= c.U && t >= 0 && t < c.T) {
                    const float lab = (lane < 31) ? nbv[j] : (j + 1 < J ? nbv[j + 1] : -INFINITY);
                    put_info(p, c, t, u, v[j], sp[(3 * J + j) * 32 + lane], sp[j * 32 + lane],
                             sp[(J + j) * 32 + lane], sp[(2 * J + j) * 32 + lane],
                             sc[(3 * J + j) * 32 + lane], lab, KA, KB);
                }
            }
        }
        // Commit diagonal d.
        Oh4 = Oh3;
        Oh3 = Oh2;
        Oh2 = O;
        O = Onew;
        {
            const int64_t base = c.off + diag_start(d, c.T, c.W) - max(0, d - c.U) + d;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int u = lane + 32 * j, t = d - u;
                v[j] = nv[j];
                if (u <= c.U && t >= 0 && t < c.T) p.va[base - u] = nv[j];
            }
            if (lane == 0) p.oa[c.off + d] = O;
        }
        mC = mB;
        mB = mA;
        mA = m_prev;
    }
    // Last diagonal D-1 holds only the terminal node (T-1, U).
    const int e = c.D - 1;
    const float* sp = ring + (e % R) * SL;
    const int jU = c.U >> 5, lU = c.U & 31;
    float vU = -INFINITY, lpbU = -INFINITY, vbU = -INFINITY, lseU = 0.0f;
#pragma unroll
    for (int j = 0; j < J; ++j)
        if (j == jU) {
            vU = v[j];
            lpbU = sp[j * 32 + lane];
            vbU = sp[(3 * J + j) * 32 + lane];
            lseU = sp[(2 * J + j) * 32 + lane];
        }
    if (lane == lU) {
        if (comb_on && e > c.dm) {
            const int Qe = __float_as_int(sp[4 * J * 32 + lane]);
            put_info(p, c, c.T - 1, c.U, vU, vbU, lpbU, -INFINITY, lseU, 0.0f, -INFINITY,
                     (float)(O + Qe - C), (float)(O - C));
        }
        const double ll2 = (double)O + (double)vU + (double)lpbU;
        p.lossa[c.b] = -ll2 * kLn2;
        p.loss[c.b] = (float)(-ll2 * kLn2);
        p.delta[c.b] = (float)((double)C - ll2);
    }
}

template <int J>
__device__ void dp_beta(const Params& p, const Samp& c, float* ring, int* xch) {
    constexpr int R = Ring<J>::R, PF = R - 2, SL = ring_slot_floats(J);
    const int lane = threadIdx.x & 31;
    float v[J];   // beta of diagonal d+1 (virtual diagonal D: 0 at column U)
#pragma unroll
    for (int j = 0; j < J; ++j) v[j] = (lane + 32 * j == c.U) ? 0.0f : -INFINITY;
    for (int k = 0; k <= PF; ++k) {
        ring_issue<J>(c, ring, c.D - 1 - k, false, p.lpb, p.lpy, p.lse2, p.va, p.oa, lane);
        cp_commit();
    }
    int Q = 0, Qh2 = 0, Qh3 = 0, Qh4 = 0;   // frames of d+1..d+4 (mirror of dp_alpha)
    float mA = -INFINITY, mB = -INFINITY, mC = -INFINITY;
    bool synced = false;
    int C = 0;
    const bool comb_on = p.want_grad != 0;

    for (int d = c.D - 1; d >= 0; --d) {
        if (d == c.dm) {
            if (lane == 0) xch[1] = Q;   // frame of diagonal dm+1
            asm volatile("bar.sync 1, 64;\n" ::: "memory");
            C = xch[0] + xch[1];
            synced = true;
            if (comb_on) {
                for (int e = c.dm; e >= max(0, c.dm - PF); --e) {
                    float* sl = ring + (e % R) * SL;
                    const int64_t base = c.off + diag_start(e, c.T, c.W) - max(0, e - c.U) + e;
#pragma unroll
                    for (int j = 0; j < J; ++j) {
                        const int u = lane + 32 * j, t = e - u;
                        float* q = sl + j * 32 + lane;
                        if (u <= c.U && t >= 0 && t < c.T) {
                            cp4(q + 2 * J * 32, p.lse2 + base - u);
                            cp4(q + 3 * J * 32, p.va + base - u);
                        } else {
                            q[2 * J * 32] = 0.0f;
                            q[3 * J * 32] = -INFINITY;
                        }
                    }
                    cp4(sl + 4 * J * 32 + lane, p.oa + c.off + e);
                }
                cp_commit();
                cp_wait_all();
            }
        }
        ring_issue<J>(c, ring, d - PF - 1, synced && comb_on, p.lpb, p.lpy, p.lse2, p.va, p.oa,
                      lane);
        cp_commit();
        cp_wait<PF + 1>();
        __syncwarp();
        const float* sd = ring + (d % R) * SL;

        int Qnew = Q;
        if (fabsf(mB) < 1e6f && fabsf(mC) < 1e6f) {
            const int b3 = Qh3 + (int)rintf(mB), b4 = Qh4 + (int)rintf(mC);
            Qnew = b3 + 3 * (b3 - b4);
        }
        const int tau = Qnew - Q;
        const float sh = (float)tau;
        float nbv[J], nv[J], lab[J];
#pragma unroll
        for (int j = 0; j < J; ++j) nbv[j] = __shfl_sync(0xffffffffu, v[j], (lane + 1) & 31);
#pragma unroll
        for (int j = 0; j < J; ++j) {
            lab[j] = (lane < 31) ? nbv[j] : (j + 1 < J ? nbv[j + 1] : -INFINITY);
            nv[j] = lae2(v[j] + (sd[j * 32 + lane] - sh), lab[j] + (sd[(J + j) * 32 + lane] - sh));
        }
        const float m_next = warp_max_valid<J>(v, d + 1, c, lane);
        const int Qn = Q;   // frame of d+1
        Qh4 = Qh3;
        Qh3 = Qh2;
        Qh2 = Q;
        Q = Qnew;           // frame of d

        if (synced && comb_on) {
            const int Oe = __float_as_int(sd[4 * J * 32 + lane]);
            const float KA = (float)(Oe + Q - C), KB = (float)(Oe + Qn - C);
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int u = lane + 32 * j, t = d - u;
                if (u <= c.U && t >= 0 && t < c.T)
                    put_info(p, c, t, u, sd[(3 * J + j) * 32 + lane], nv[j], sd[j * 32 + lane],
                             sd[(J + j) * 32 + lane], sd[(2 * J + j) * 32 + lane], v[j], lab[j],
                             KA, KB);
            }
        }
        {
            const int64_t base = c.off + diag_start(d, c.T, c.W) - max(0, d - c.U) + d;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int u = lane + 32 * j, t = d - u;
                v[j] = nv[j];
                if (u <= c.U && t >= 0 && t < c.T) p.vb[base - u] = nv[j];
            }
            if (lane == 0) p.qb[c.off + d] = Q;
        }
        mC = mB;
        mB = mA;
        mA = m_next;
    }
    if (lane == 0) p.lossb[c.b] = -((double)Q + (double)v[0]) * kLn2;
}

template <int J>
__device__ __forceinline__ void dp_run(const Params& p, const Samp& c, float* ring, int* xch) {
    if (threadIdx.x < 32) dp_alpha<J>(p, c, ring, xch);
    else dp_beta<J>(p, c, ring + p.ring_floats, xch);
}

__global__ void __launch_bounds__(64) k_dp(Params p) {
    if (*p.err) return;
    extern __shared__ float smem[];
    __shared__ int xch[2];
    Samp c;
    c.b = p.order[blockIdx.x];
    c.T = p.Tl[c.b];
    c.U = p.Ul[c.b];
    c.W = c.U + 1;
    c.D = c.T + c.U;
    c.dm = (c.D - 1) / 2;
    c.off = p.off[c.b];
    const int J = (c.W + 31) >> 5;
    if (J <= 1) dp_run<1>(p, c, smem, xch);
    else if (J <= 2) dp_run<2>(p, c, smem, xch);
    else if (J <= 4) dp_run<4>(p, c, smem, xch);
    else if (J <= 8) dp_run<8>(p, c, smem, xch);
    else if (J <= 16) dp_run<16>(p, c, smem, xch);
    else dp_run<32>(p, c, smem, xch);
}

// ---------------------------------------------------------------- grad pass
template <typename Tin, int G, bool VEC, bool FUSED>
__global__ void __launch_bounds__(256) k_grad(Params p) {
    if (*p.err) return;
    using E = Elt<Tin>;
    const Tin* X = static_cast<const Tin*>(p.logits);
    Tin* Y = static_cast<Tin*>(p.grad);
    const int V = p.V;
    const int lane = threadIdx.x & (G - 1);
    const int64_t ng = (int64_t)gridDim.x * (blockDim.x / G);
    const float cl = p.clamp, sc = p.scale;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / G; r < p.rows; r += ng) {
        const int b = find_sample(p.off, p.B, r);
        const int y = row_label(p, b, r);
        const float4 in = p.info[r];
        const float dl = __ldg(p.delta + b);
        const Tin* row = X + r * (int64_t)V;
        Tin* out = Y + r * (int64_t)V;
        const bool zero = (in.y + dl) < p.skip2;
        const float w2 = in.x + dl;
        const float eb = zero ? 0.0f : ex2(in.z + dl);
        const float ey = zero ? 0.0f : ex2(in.w + dl);
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
                    g[e] = fminf(fmaxf(gv, -cl), cl) * sc;
                }
                __stcs(ov + vi, E::pack(g));
            }
        } else {
            for (int k = lane; k < V; k += G) {
                float gv = (FUSED && !zero) ? ex2(fmaf(E::to_f(row[k]), kLog2e, w2)) : 0.0f;
                if (k == p.blank) gv -= eb;
                if (k == y) gv -= ey;
                out[k] = E::from_f(fminf(fmaxf(gv, -cl), cl) * sc);
            }
        }
    }
}

// ---------------------------------------------------------------- finalize
__global__ void __launch_bounds__(256) k_finalize(Params p) {
    __shared__ double part[256];
    __shared__ int errs;
    const int tid = threadIdx.x;
    if (tid == 0) errs = *p.err;
    __syncthreads();
    const bool ok_in = errs == 0;
    double s = 0.0;
    if (ok_in) {
        for (int b = tid; b < p.B; b += blockDim.x) {
            const double la = p.lossa[b], lb = p.lossb[b];
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
        if (ok_in && p.loss_red) p.loss_red[0] = (float)(p.red == RNNT_RED_MEAN ? part[0] / p.B : part[0]);
        int st = RNNT_OK;
        if (errs & (ERR_LENGTH | ERR_ROWS | ERR_TARGET)) st = RNNT_INVALID_VALUE;
        else if (errs & ERR_MISMATCH) st = RNNT_LOSS_MISMATCH;
        *p.err = errs;
        if (p.status) *p.status = st;
    }
}

// ---------------------------------------------------------------- grad scale
template <typename Tin>
__global__ void __launch_bounds__(256) k_scale(void* grad, int64_t rows, int V, int B,
                                               const int64_t* off, const float* factors,
                                               int per_sample) {
    if (!per_sample && factors[0] == 1.0f) return;
    using E = Elt<Tin>;
    Tin* G = static_cast<Tin*>(grad);
    const int64_t ng = (int64_t)gridDim.x * (blockDim.x / 32);
    const int lane = threadIdx.x & 31;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32; r < rows; r += ng) {
        const float f = per_sample ? factors[find_sample(off, B, r)] : factors[0];
        if (f == 1.0f) continue;
        Tin* row = G + r * (int64_t)V;
        for (int k = lane; k < V; k += 32) row[k] = E::from_f(E::to_f(row[k]) * f);
    }
}

// ---------------------------------------------------------------- host side
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

int ring_floats_for(int S) {
    const int W = S + 1;
    const int Jn = (W + 31) / 32;
    int best = 0;
    const int Js[6] = {1, 2, 4, 8, 16, 32};
    const int Rs[6] = {32, 32, 16, 8, 6, 4};
    for (int i = 0; i < 6; ++i) {
        const int need = Rs[i] * ring_slot_floats(Js[i]);
        if (need > best) best = need;
        if (Js[i] >= Jn) break;
    }
    return best;
}

template <typename Tin>
void launch_rows(const Params& p, cudaStream_t st, int sms) {
    const int V = p.V;
    const bool vec = ((size_t)V * sizeof(Tin)) % 16 == 0;
    const int64_t need_threads = p.rows * 32;
    int64_t blocks = (need_threads + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;
    const int grid = (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
    if (!p.fused) {
        int64_t gb = (p.rows + 255) / 256;
        const int g2 = (int)(gb < cap ? (gb > 0 ? gb : 1) : cap);
        k_row_gather<Tin><<<g2, 256, 0, st>>>(p);
        return;
    }
#define ROWK(G_)                                                                   \
    do {                                                                           \
        if (vec) k_row_fused<Tin, G_, true><<<grid, 256, 0, st>>>(p);              \
        else k_row_fused<Tin, G_, false><<<grid, 256, 0, st>>>(p);                 \
    } while (0)
    if (V >= 512) ROWK(32);
    else if (V >= 128) ROWK(16);
    else if (V >= 32) ROWK(8);
    else ROWK(4);
#undef ROWK
}

template <typename Tin>
void launch_grad(const Params& p, cudaStream_t st, int sms) {
    const int V = p.V;
    const bool vec = ((size_t)V * sizeof(Tin)) % 16 == 0;
    const int64_t cap = (int64_t)sms * 8;
    const int64_t blocks = (p.rows * 32 + 255) / 256;
    const int grid = (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
#define GRADK(G_)                                                                          \
    do {                                                                                   \
        if (p.fused) {                                                                     \
            if (vec) k_grad<Tin, G_, true, true><<<grid, 256, 0, st>>>(p);                 \
            else k_grad<Tin, G_, false, true><<<grid, 256, 0, st>>>(p);                    \
        } else {                                                                           \
            if (vec) k_grad<Tin, G_, true, false><<<grid, 256, 0, st>>>(p);                \
            else k_grad<Tin, G_, false, false><<<grid, 256, 0, st>>>(p);                   \
        }                                                                                  \
    } while (0)
    if (V >= 512) GRADK(32);
    else if (V >= 128) GRADK(16);
    else if (V >= 32) GRADK(8);
    else GRADK(4);
#undef GRADK
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

}  // namespace

extern "C" rnnt_status_t rnnt_workspace_size(int32_t B, int64_t rows, int32_t V, rnnt_dtype_t dt,
                                             size_t* bytes) {
    if (!bytes || B < 1 || rows < 1 || V < 1 || (dt != RNNT_F32 && dt != RNNT_F16))
        return RNNT_INVALID_VALUE;
    *bytes = ws_layout(B, rows).total;
    return RNNT_OK;
}

extern "C" rnnt_status_t rnnt_loss_fused_staged(
    const void* logits, rnnt_dtype_t dt, int64_t rows, int32_t V, const int32_t* targets,
    int32_t targets_stride, const int32_t* logit_lengths, const int32_t* target_lengths, int32_t B,
    int32_t blank, float clamp, int32_t fused_log_softmax, rnnt_reduction_t reduction, float* loss,
    float* loss_reduced, void* grad, void* workspace, size_t workspace_bytes, int32_t* status_dev,
    rnnt_stream_t stream, void* const* stage_events) {
    if (!logits || !targets || !logit_lengths || !target_lengths || !loss || !workspace)
        return RNNT_INVALID_VALUE;
    if (dt != RNNT_F32 && dt != RNNT_F16) return RNNT_INVALID_VALUE;
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
    if (workspace_bytes < L.total) return RNNT_WORKSPACE_TOO_SMALL;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RNNT_LAUNCH_FAILED;
    const int sms = num_sms(dev);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    char* w = static_cast<char*>(workspace);
    Params p;
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
    // smallest subnormal of the output type, so it rounds to zero.
    const float zero_at = dt == RNNT_F16 ? -25.5f : -151.0f;
    p.skip2 = zero_at - log2f(p.scale);
    p.fused = fused_log_softmax ? 1 : 0;
    p.red = reduction;
    p.want_grad = grad != nullptr;
    p.ring_floats = ring_floats_for(targets_stride);
    p.loss = loss;
    p.loss_red = loss_reduced;
    p.status = status_dev;
    p.err = reinterpret_cast<int32_t*>(w + L.err);
    p.off = reinterpret_cast<int64_t*>(w + L.off);
    p.order = reinterpret_cast<int32_t*>(w + L.order);
    p.lossa = reinterpret_cast<double*>(w + L.lossa);
    p.lossb = reinterpret_cast<double*>(w + L.lossb);
    p.delta = reinterpret_cast<float*>(w + L.delta);
    p.lse2 = reinterpret_cast<float*>(w + L.lse2);
    p.lpb = reinterpret_cast<float*>(w + L.lpb);
    p.lpy = reinterpret_cast<float*>(w + L.lpy);
    p.va = reinterpret_cast<float*>(w + L.va);
    p.vb = reinterpret_cast<float*>(w + L.vb);
    p.oa = reinterpret_cast<int32_t*>(w + L.oa);
    p.qb = reinterpret_cast<int32_t*>(w + L.qb);
    p.info = reinterpret_cast<float4*>(w + L.info);

    const size_t dp_smem = (size_t)p.ring_floats * 2 * sizeof(float);
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
    mark(0);
    k_prepare<<<1, 1024, 0, st>>>(p);
    mark(1);
    if (dt == RNNT_F32) launch_rows<float>(p, st, sms);
    else launch_rows<__half>(p, st, sms);
    mark(2);
    k_dp<<<B, 64, dp_smem, st>>>(p);
    mark(3);
    if (grad) {
        if (dt == RNNT_F32) launch_grad<float>(p, st, sms);
        else launch_grad<__half>(p, st, sms);
    }
    mark(4);
    k_finalize<<<1, 256, 0, st>>>(p);
    mark(5);
    return cudaGetLastError() == cudaSuccess ? RNNT_OK : RNNT_LAUNCH_FAILED;
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
    if (dt != RNNT_F32 && dt != RNNT_F16) return RNNT_INVALID_VALUE;
    const Layout L = ws_layout(B, rows);
    if (workspace_bytes < L.total) return RNNT_WORKSPACE_TOO_SMALL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RNNT_LAUNCH_FAILED;
    const int64_t cap = (int64_t)num_sms(dev) * 8;
    const int64_t blocks = (rows * 32 + 255) / 256;
    const int grid = (int)(blocks < cap ? blocks : cap);
    const int64_t* off = reinterpret_cast<const int64_t*>(static_cast<const char*>(workspace) + L.off);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (dt == RNNT_F32) k_scale<float><<<grid, 256, 0, st>>>(grad, rows, V, B, off, factors, per_sample);
    else k_scale<__half><<<grid, 256, 0, st>>>(grad, rows, V, B, off, factors, per_sample);
    return cudaGetLastError() == cudaSuccess ? RNNT_OK : RNNT_LAUNCH_FAILED;
}

extern "C" const char* rnnt_status_string(rnnt_status_t s) {
    switch (s) {
        case RNNT_OK: return "success";
        case RNNT_INVALID_VALUE: return "invalid value (arguments, lengths or targets)";
        case RNNT_WORKSPACE_TOO_SMALL: return "workspace too small";
        case RNNT_LAUNCH_FAILED: return "kernel launch failed";
        case RNNT_LOSS_MISMATCH: return "alpha/beta loss mismatch or non-finite loss";
        case RNNT_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

extern "C" int32_t rnnt_abi_version(void) { return 100; }
