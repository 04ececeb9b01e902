// common.cuh -- definitions shared by the translation units of the rejection sampler
// (sm_103a): the workspace plan and kernel parameters, element access, warp reductions,
// the TMA bulk-copy primitives, the per-chunk softmax / argmax partials and the
// inverse-CDF search.  Everything but the shared types has internal linkage.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <limits.h>
#include <math.h>

#include "spec_reject.h"

namespace specrej {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
#ifndef SPEC_UNIT_BYTES
#define SPEC_UNIT_BYTES 8192
#endif
#ifndef SPEC_LDG_UNROLL
#define SPEC_LDG_UNROLL 4       // 16-byte vectors in flight per lane (register-staged K1)
#endif
#ifndef SPEC_LDG_MIN_BLOCKS
#define SPEC_LDG_MIN_BLOCKS 3   // blocks of 256 per SM the register-staged K1 must fit
#endif
constexpr int kUnitBytes = SPEC_UNIT_BYTES;  // bytes of logits per (row, chunk) unit
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

// Layout of the workspace (all offsets 256-byte aligned).  The error word comes first so
// that spec_reject_last_device_error() finds it without knowing the call's sizes.
struct Plan {
    int chunk;    // logits per chunk
    int nchunks;  // chunks per row
    size_t off_err, off_part, off_rstate, off_rstat, off_rpart, off_rcnt, off_thr, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline bool make_plan(int32_t B, int64_t T, int32_t V, spec_dtype dt, int has_q, Plan *pl)
{
    if (B < 0 || T < 0 || V < 1 || V > SPEC_REJECT_MAX_VOCAB || (dt != SPEC_F32 && dt != SPEC_BF16))
        return false;
    const int es = dt == SPEC_BF16 ? 2 : 4;
    pl->chunk = kUnitBytes / es;
    pl->nchunks = (V + pl->chunk - 1) / pl->chunk;
    size_t o = 0;
    pl->off_err = o;
    o = align256(o + 4 * sizeof(int32_t));
    pl->off_part = o;
    o = align256(o + sizeof(float2) * (size_t)T * (size_t)pl->nchunks);
    pl->off_rstate = o;
    o = align256(o + sizeof(int32_t) * (size_t)(B + 1));
    pl->off_rstat = o;
    o = align256(o + sizeof(float2) * (size_t)(B + 1));
    pl->off_rpart = o;
    o = align256(o + (has_q ? sizeof(float) * (size_t)B * (size_t)pl->nchunks : 0));
    pl->off_rcnt = o;
    o = align256(o + (has_q ? sizeof(int32_t) * (size_t)B : 0));
    pl->off_thr = o;
    o = align256(o + sizeof(uint32_t) * (size_t)T);
    pl->total = o + 256;  // slack for aligning the caller's pointer
    return true;
}

struct Params {
    const void *logits;
    int64_t T;
    int32_t V;
    int64_t lstride;  // elements
    const float *q;
    int64_t qstride;  // elements
    const int32_t *ids;
    const int32_t *cu;
    int32_t B;
    const float *uni;
    const float *temp;
    int32_t *out_tokens;
    int32_t *out_acc;
    // workspace
    float2 *part;     // [T * nchunks] chunk partials
    int32_t *err;     // [0] SPEC_DEVERR_* bits, [1] first bad request (INT_MAX = none)
    int32_t *rstate;  // [B] output position j of a pending explicit-q recovery, else -1
    float2 *rstat;    // [B] (M, S) of that output row
    float *rpart;     // [B * nchunks] residual chunk masses
    int32_t *rcnt;    // [B] residual chunks done (zeroed by K2, counted up by K3)
    int chunk, nchunks;
    // top-k / top-p restriction of the target (all null without filters)
    const int32_t *top_k;  // [B]
    const float *top_p;    // [B]
    unsigned long long *counters;  // [SPEC_METRIC_COUNT] acceptance counters to add to, or null
    uint32_t *thr;         // [T] order key below which a token is cut (0 = none)
    // rows read from host memory by KL: device copies of the target rows it streams ([T, lstride],
    // written only where read) and of the draft rows its residual passes read ([T - B, V])
    char *lstage;
    float *qstage;
    // diagnostics (all may be null)
    float *dbg_pdraft;
    float *dbg_z;
    // first-rejection pass: the requests [r_begin, r_end) this launch serves, and the index of
    // its request counter in the error word; wait_prior = 0 for a launch chained after another
    // pass launch whose results it does not read (it starts as that launch's blocks finish)
    int32_t r_begin, r_end, qslot, wait_prior;
};


namespace {

// ---------------------------------------------------------------------------------------
// Element access
// ---------------------------------------------------------------------------------------

template <int DT> struct Elem;
template <> struct Elem<0> {  // fp32
    static constexpr int kVec = 4;
    static constexpr int kSize = 4;
};
template <> struct Elem<1> {  // bf16
    static constexpr int kVec = 8;
    static constexpr int kSize = 2;
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Streaming 16-byte load through the non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

template <int DT> __device__ __forceinline__ void unpack(const uint4 &w, float *x);
template <> __device__ __forceinline__ void unpack<0>(const uint4 &w, float *x)
{
    x[0] = __uint_as_float(w.x);
    x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z);
    x[3] = __uint_as_float(w.w);
}
template <> __device__ __forceinline__ void unpack<1>(const uint4 &w, float *x)
{
    x[0] = __uint_as_float(w.x << 16);
    x[1] = __uint_as_float(w.x & 0xffff0000u);
    x[2] = __uint_as_float(w.y << 16);
    x[3] = __uint_as_float(w.y & 0xffff0000u);
    x[4] = __uint_as_float(w.z << 16);
    x[5] = __uint_as_float(w.z & 0xffff0000u);
    x[6] = __uint_as_float(w.w << 16);
    x[7] = __uint_as_float(w.w & 0xffff0000u);
}

template <int DT> __device__ __forceinline__ uint4 neg_inf_vec();
template <> __device__ __forceinline__ uint4 neg_inf_vec<0>() { return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u); }
template <> __device__ __forceinline__ uint4 neg_inf_vec<1>() { return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u); }

template <int DT> __device__ __forceinline__ float load1(const char *row, int64_t v);
template <> __device__ __forceinline__ float load1<0>(const char *row, int64_t v)
{
    return __ldg(reinterpret_cast<const float *>(row) + v);
}
template <> __device__ __forceinline__ float load1<1>(const char *row, int64_t v)
{
    const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(row) + v);
    return __uint_as_float(uint32_t(b) << 16);
}

// Order-preserving unsigned key of a logit (bf16: 16 bits, fp32: 32 bits): a < b iff
// key(a) < key(b), and a == b (-0 == +0) iff the keys are equal, for non-NaN values.  The
// key is 0x8000.. plus the signed magnitude, so every key is at least 1.
template <int DT> __device__ __forceinline__ uint32_t key_of(float x);
template <> __device__ __forceinline__ uint32_t key_of<0>(float x)
{
    const uint32_t b = __float_as_uint(x);
    const uint32_t s = (uint32_t)((int32_t)b >> 31);
    return 0x80000000u + (((b & 0x7fffffffu) ^ s) - s);
}
template <> __device__ __forceinline__ uint32_t key_of<1>(float x)
{
    const uint32_t b = __float_as_uint(x);
    const uint32_t s = (uint32_t)((int32_t)b >> 31);
    return 0x8000u + ((((b >> 16) & 0x7fffu) ^ s) - s);
}

// The logit whose order key is `key` (inverse of key_of; -0 comes back as +0).
template <int DT> __device__ __forceinline__ float x_of(uint32_t key);
template <> __device__ __forceinline__ float x_of<0>(uint32_t key)
{
    return __uint_as_float(key >= 0x80000000u ? key - 0x80000000u : 0x80000000u | (0x80000000u - key));
}
template <> __device__ __forceinline__ float x_of<1>(uint32_t key)
{
    return __uint_as_float((key >= 0x8000u ? key - 0x8000u : 0x8000u | (0x8000u - key)) << 16);
}

// Whether a token survives the row's top-k / top-p cut.  F: the call has cuts (thr = 0 on a
// row keeps everything, every key being at least 1); without cuts the test compiles away.
template <int DT, bool F> __device__ __forceinline__ bool kept(float x, uint32_t thr)
{
    return !F || key_of<DT>(x) >= thr;
}

template <int DT> __device__ __forceinline__ const char *row_ptr(const Params &P, int64_t t)
{
    return reinterpret_cast<const char *>(P.logits) + t * P.lstride * Elem<DT>::kSize;
}

// ---------------------------------------------------------------------------------------
// Warp reductions (fixed butterfly order: deterministic)
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Inclusive prefix sum over lanes (Kogge-Stone, fixed order).
__device__ __forceinline__ float warp_incl_scan(float v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(kFull, v, o);
        if (lane >= o)
            v += n;
    }
    return v;
}

// Largest value, lowest index on ties.
__device__ __forceinline__ void warp_argmax(float &best, int &idx)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float b2 = __shfl_xor_sync(kFull, best, o);
        const int i2 = __shfl_xor_sync(kFull, idx, o);
        if (b2 > best || (b2 == best && i2 < idx)) {
            best = b2;
            idx = i2;
        }
    }
}

// ---------------------------------------------------------------------------------------
// K1: row statistics
// ---------------------------------------------------------------------------------------

// Running softmax statistics of one lane: max m (raw logit), reference M = fl(m * c) and
// s = sum 2^(l * c - M).
struct SoftAcc {
    float m = -INFINITY, M = -INFINITY, s = 0.f;
    __device__ __forceinline__ void rebase(float bm, float c)
    {
        if (bm > m) {
            const float Mn = bm * c;
            s = (m == -INFINITY) ? 0.f : s * ex2(M - Mn);
            m = bm;
            M = Mn;
        }
    }
};

struct ArgAcc {
    float best = -INFINITY;
    int idx = INT_MAX;
    __device__ __forceinline__ void add(float x, int v)
    {
        if (x > best) {
            best = x;
            idx = v;
        }
    }
};

// Block 0 of K1: check the ragged layout, initialise the error word.
__device__ void validate_layout(const Params &P)
{
    __shared__ int s_first;
    if (threadIdx.x == 0)
        s_first = INT_MAX;
    __syncthreads();
    int layout_bad = 0, len_bad = 0;
    for (int r = threadIdx.x; r < P.B; r += blockDim.x) {
        const int k = P.cu[r + 1] - P.cu[r];
        if (k < 0)
            layout_bad = 1;
        if (k > SPEC_REJECT_MAX_SPEC_LEN) {
            len_bad = 1;
            atomicMin(&s_first, r);
        }
    }
    if (threadIdx.x == 0 && (P.cu[0] != 0 || (int64_t)P.cu[P.B] + P.B != P.T))
        layout_bad = 1;
    layout_bad = __syncthreads_or(layout_bad);
    len_bad = __syncthreads_or(len_bad);
    if (threadIdx.x == 0) {
        P.err[0] = (layout_bad ? SPEC_DEVERR_LAYOUT : 0) | (len_bad ? SPEC_DEVERR_SPEC_LEN : 0);
        P.err[1] = layout_bad ? -1 : s_first;
    }
}

// Request that owns target row t (rows are request-major; cu[r] + r is increasing for a
// valid layout; for an invalid one any in-range answer is fine, K2 reports the error).
__device__ __forceinline__ int find_request(const Params &P, int64_t t)
{
    int lo = 0, hi = P.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)__ldg(P.cu + mid) + mid <= t)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Bounds of one (row, chunk) unit: 16-byte aligned body [vlo, vlo + nvec * VEC) and
// scalar head [lo, vlo) and tail [vhi, hi), each shorter than one vector.
struct UnitRange {
    int64_t lo, hi, vlo, nvec, vhi;
};

template <int DT> __device__ __forceinline__ UnitRange unit_range(const Params &P, const char *row, int c)
{
    constexpr int VEC = Elem<DT>::kVec;
    constexpr int ES = Elem<DT>::kSize;
    UnitRange R;
    R.lo = (int64_t)c * P.chunk;
    R.hi = min((int64_t)P.V, R.lo + P.chunk);
    const uintptr_t a = reinterpret_cast<uintptr_t>(row + R.lo * ES);
    R.vlo = min(R.hi, R.lo + (int64_t)(((16 - (a & 15)) & 15) / ES));
    R.nvec = (R.hi - R.vlo) / VEC;
    R.vhi = R.vlo + R.nvec * VEC;
    return R;
}

// Largest of the elements of a vector (bf16: packed max on the raw pairs).
template <int DT> __device__ __forceinline__ float vec_max(const uint4 &w);
template <> __device__ __forceinline__ float vec_max<0>(const uint4 &w)
{
    return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)), fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
}
template <> __device__ __forceinline__ float vec_max<1>(const uint4 &w)
{
    uint32_t a, b, m;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(w.x), "r"(w.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(w.z), "r"(w.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
}

// Source of the 16-byte vectors of a unit body: streaming loads from global memory.
struct GlobalVec {
    static constexpr int kUnroll = SPEC_LDG_UNROLL;  // vectors in flight per lane
    const char *base;
    __device__ __forceinline__ uint4 operator()(int64_t vi) const { return ld_stream(base + vi * 16); }
};

// Softmax partial of one unit: body vectors from `src`, head / tail scalars from `row`.
template <int DT, class SRC>
__device__ __forceinline__ void softmax_body(const Params &P, int64_t t, int c, float cs, int lane, const SRC &src,
                                             const UnitRange &R, const char *row)
{
    constexpr int VEC = Elem<DT>::kVec;
    const int64_t lo = R.lo, hi = R.hi, vlo = R.vlo, nvec = R.nvec, vhi = R.vhi;
    {
        SoftAcc acc;
        float sacc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            sacc[e] = 0.f;
        for (int64_t b0 = 0; b0 < nvec; b0 += 32 * SRC::kUnroll) {
            uint4 raw[SRC::kUnroll];
#pragma unroll
            for (int u = 0; u < SRC::kUnroll; ++u) {
                const int64_t vi = b0 + u * 32 + lane;
                raw[u] = (vi < nvec) ? src(vi) : neg_inf_vec<DT>();
            }
            float bm = -INFINITY;
#pragma unroll
            for (int u = 0; u < SRC::kUnroll; ++u)
                bm = fmaxf(bm, vec_max<DT>(raw[u]));
            if (bm > acc.m) {
                // fold the per-slot sums into the lane sum before moving the reference
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    s += sacc[e];
                    sacc[e] = 0.f;
                }
                acc.s += s;
                acc.rebase(bm, cs);
            }
            if (acc.m > -INFINITY) {  // nothing but -inf so far: no mass, and M is not finite
                const float M = acc.M;
#pragma unroll
                for (int u = 0; u < SRC::kUnroll; ++u) {
                    float x[VEC];
                    unpack<DT>(raw[u], x);
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        sacc[e] += ex2(fmaf(x[e], cs, -M));
                }
            }
        }
        {
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                s += sacc[e];
            acc.s += s;
        }
        // scalar head and tail (fewer than VEC elements each)
        float xh = -INFINITY, xt = -INFINITY;
        if (lane < vlo - lo)
            xh = load1<DT>(row, lo + lane);
        if (lane < hi - vhi)
            xt = load1<DT>(row, vhi + lane);
        const float bm = fmaxf(xh, xt);
        if (bm > -INFINITY) {
            acc.rebase(bm, cs);
            acc.s += ex2(fmaf(xh, cs, -acc.M)) + ex2(fmaf(xt, cs, -acc.M));
        }
        // warp combine
        const float mw = warp_max(acc.m);
        const float Mw = mw * cs;
        const float sl = (acc.m == -INFINITY) ? 0.f : acc.s * ex2(acc.M - Mw);
        const float sw = warp_sum(sl);
        if (lane == 0)
            P.part[t * P.nchunks + c] = make_float2(mw, mw == -INFINITY ? 0.f : sw);
    }
}

// Argmax partial of one unit (greedy rows).
template <int DT, class SRC>
__device__ __forceinline__ void argmax_body(const Params &P, int64_t t, int c, int lane, const SRC &src,
                                            const UnitRange &R, const char *row)
{
    constexpr int VEC = Elem<DT>::kVec;
    const int64_t lo = R.lo, hi = R.hi, vlo = R.vlo, nvec = R.nvec, vhi = R.vhi;
    {
        ArgAcc acc;
        if (lane < vlo - lo)
            acc.add(load1<DT>(row, lo + lane), (int)(lo + lane));
        for (int64_t b0 = 0; b0 < nvec; b0 += 32 * SRC::kUnroll) {
            uint4 raw[SRC::kUnroll];
#pragma unroll
            for (int u = 0; u < SRC::kUnroll; ++u) {
                const int64_t vi = b0 + u * 32 + lane;
                if (vi < nvec)
                    raw[u] = src(vi);
            }
#pragma unroll
            for (int u = 0; u < SRC::kUnroll; ++u) {
                const int64_t vi = b0 + u * 32 + lane;
                if (vi < nvec) {
                    float x[VEC];
                    unpack<DT>(raw[u], x);
                    const int v0 = (int)(vlo + vi * VEC);
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        acc.add(x[e], v0 + e);
                }
            }
        }
        if (lane < hi - vhi)
            acc.add(load1<DT>(row, vhi + lane), (int)(vhi + lane));
        warp_argmax(acc.best, acc.idx);
        if (lane == 0)
            P.part[t * P.nchunks + c] = make_float2(acc.best, __int_as_float(acc.idx));
    }
}

template <int DT> __device__ __noinline__ void softmax_unit(const Params &P, int64_t t, int c, float cs, int lane)
{
    const char *row = row_ptr<DT>(P, t);
    const UnitRange R = unit_range<DT>(P, row, c);
    softmax_body<DT>(P, t, c, cs, lane, GlobalVec{row + R.vlo * Elem<DT>::kSize}, R, row);
}

template <int DT> __device__ __noinline__ void argmax_unit(const Params &P, int64_t t, int c, int lane)
{
    const char *row = row_ptr<DT>(P, t);
    const UnitRange R = unit_range<DT>(P, row, c);
    argmax_body<DT>(P, t, c, lane, GlobalVec{row + R.vlo * Elem<DT>::kSize}, R, row);
}

template <int DT>
__device__ __forceinline__ void rowstats_unit(const Params &P, int64_t t, int c, bool greedy, float cs, int lane)
{
    if (greedy)
        argmax_unit<DT>(P, t, c, lane);
    else
        softmax_unit<DT>(P, t, c, cs, lane);
}

// Per-row parameters a unit needs: greedy or not, and c = log2(e) / T_r.
struct RowInfo {
    int64_t t = -1;
    bool greedy = true;
    float cs = 0.f;
};

// force_argmax: 0 = by temperature, 1 = argmax on every row, kArgmaxKeepErrors = argmax on
// every row of a call whose error word already holds its results (no layout check, which would
// reset the word).
constexpr int kArgmaxKeepErrors = 2;

__device__ __forceinline__ void row_info(const Params &P, int64_t t, int force_argmax, RowInfo &ri)
{
    ri.t = t;
    const float temp = __ldg(P.temp + find_request(P, t));
    ri.greedy = force_argmax || !(temp > 0.f);
    ri.cs = ri.greedy ? 0.f : kLog2e / temp;
}

// ---------------------------------------------------------------------------------------
// mbarrier and bulk-copy helpers (TMA)
// ---------------------------------------------------------------------------------------

constexpr uint32_t kWaitLimit = 1u << 22;  // polls before a wait gives up (far above any real wait)

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Orders this thread's earlier generic-proxy writes to global memory before later bulk copies
// (async proxy) that read them, once a barrier has passed.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok)
                 : "r"(smem_addr(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete, at most kWaitLimit polls.  On
// giving up it sets SPEC_DEVERR_TIMEOUT in the error word and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *err)
{
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity))
            return true;
    atomicOr(err, SPEC_DEVERR_TIMEOUT);
    return false;
}


// One bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16), its
// completion counted on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

constexpr int kVecPerLane = kUnitBytes / 16 / 32;  // 16-byte vectors of a unit held by each lane

// Softmax partial of a unit held in registers: v[k] is body vector k * 32 + lane (slots
// past the body hold -inf), the scalar tail comes from global memory.
template <int DT>
__device__ __forceinline__ void softmax_regs(float2 *out, float cs, int lane, const uint4 (&v)[kVecPerLane],
                                             const UnitRange &R, const char *row)
{
    constexpr int VEC = Elem<DT>::kVec;
    float xt = -INFINITY;
    if (lane < R.hi - R.vhi)
        xt = load1<DT>(row, R.vhi + lane);
    float m = xt;
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k)
        m = fmaxf(m, vec_max<DT>(v[k]));
    const float M = m * cs;
    float s = 0.f;
    if (m > -INFINITY) {
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            acc[e] = 0.f;
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            float x[VEC];
            unpack<DT>(v[k], x);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                acc[e] += ex2(fmaf(x[e], cs, -M));
        }
        acc[0] += ex2(fmaf(xt, cs, -M));
#pragma unroll
        for (int w = VEC / 2; w > 0; w >>= 1)
#pragma unroll
            for (int e = 0; e < w; ++e)
                acc[e] += acc[e + w];
        s = acc[0];
    }
    const float mw = warp_max(m);
    const float Mw = mw * cs;
    const float sl = (m == -INFINITY) ? 0.f : s * ex2(M - Mw);
    const float sw = warp_sum(sl);
    if (lane == 0)
        *out = make_float2(mw, mw == -INFINITY ? 0.f : sw);
}

// Greedy rows: (max, lowest index of the max) of one unit held in registers.  Two passes with
// independent operations: a max tree, then the least index equal to the warp's maximum (a
// compare-and-select chain over 128 elements would serialise on its own latency).  A unit of
// -inf only keeps the index unset (INT_MAX), as a running "x > best" scan would.
template <int DT>
__device__ __forceinline__ void argmax_regs(float2 *out, int lane, const uint4 (&v)[kVecPerLane], const UnitRange &R,
                                            const char *row)
{
    constexpr int VEC = Elem<DT>::kVec;
    const bool has_tail = lane < R.hi - R.vhi;
    const float xt = has_tail ? load1<DT>(row, R.vhi + lane) : -INFINITY;
    float m = xt;
#pragma unroll
    for (int k = 0; k < kVecPerLane; ++k)
        m = fmaxf(m, vec_max<DT>(v[k]));  // vectors past the unit hold -inf
    const float mw = warp_max(m);
    int idx = INT_MAX;
    if (DT == 1 && mw > -INFINITY && mw != 0.f) {
        // bf16: a token equals the maximum iff its bits do (not for +-0, handled below).  Per
        // word, the halves where bits ^ max is zero: (d - 0x00010001) & ~d & 0x80008000 marks the
        // lower zero half exactly and can only mark the upper one falsely when the lower is zero,
        // so the first marked half of the first marked word is the vector's first maximum.
        const uint32_t mb = __float_as_uint(mw) >> 16;
        const uint32_t m2 = mb | (mb << 16);
        auto zero_halves = [&](uint32_t x) {
            const uint32_t d = x ^ m2;
            return (d - 0x00010001u) & ~d & 0x80008000u;
        };
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            const uint32_t h[4] = {zero_halves(v[k].x), zero_halves(v[k].y), zero_halves(v[k].z), zero_halves(v[k].w)};
            if (h[0] | h[1] | h[2] | h[3]) {
                const int v0 = (int)(R.vlo + ((int64_t)k * 32 + lane) * VEC);
                int e = 0;
#pragma unroll
                for (int q = 3; q >= 0; --q)
                    if (h[q])
                        e = 2 * q + ((h[q] & 0x8000u) ? 0 : 1);
                idx = min(idx, v0 + e);
            }
        }
        if (xt == mw)
            idx = min(idx, (int)(R.vhi + lane));
    } else if (mw > -INFINITY) {
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            float x[VEC];
            unpack<DT>(v[k], x);
            const int v0 = (int)(R.vlo + ((int64_t)k * 32 + lane) * VEC);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                idx = min(idx, x[e] == mw ? v0 + e : INT_MAX);
        }
        if (xt == mw)
            idx = min(idx, (int)(R.vhi + lane));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        idx = min(idx, __shfl_xor_sync(kFull, idx, o));
    if (lane == 0)
        *out = make_float2(mw, __int_as_float(idx));
}

// ---------------------------------------------------------------------------------------
// Inverse-CDF locate: chunk scan + three-level warp descent inside the chunk
// ---------------------------------------------------------------------------------------

// Mass of the target distribution in units of 2^M: w(v) = 2^(l_v c - M), x* optionally left out.
#ifndef SPEC_RANGE_UNROLL
#define SPEC_RANGE_UNROLL 8  // 16-byte groups in flight per lane in a segment sum of the draw's search
#endif
constexpr int kRangeUnroll = SPEC_RANGE_UNROLL;

// Sum of f.one(v) over [v0, v1) in index order, the elements of up to eight at a time loaded
// together (one round trip to memory instead of one per element; the additions keep their order).
template <class F> __device__ __forceinline__ float scalar_sum(const F &f, int64_t v0, int64_t v1)
{
    float tail = 0.f;
    for (int64_t v = v0; v < v1; v += 8) {
        float w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            w[e] = (v + e < v1) ? f.one(v + e) : 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (v + e < v1)
                tail += w[e];
    }
    return tail;
}

template <int DT, bool F> struct TargetMass {
    const char *row;
    float cs, M;
    int64_t excl;
    uint32_t thr;  // top-k / top-p cut of the row (0 = none)
    __device__ __forceinline__ float one(int64_t v) const
    {
        const float x = load1<DT>(row, v);
        return (v == excl || !kept<DT, F>(x, thr)) ? 0.f : ex2(fmaf(x, cs, -M));
    }
    // Sum of masses of elements [v0, v1); vector loads where the row is 16-byte aligned.
    __device__ __forceinline__ float range(int64_t v0, int64_t v1) const
    {
        constexpr int VEC = Elem<DT>::kVec;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        int64_t v = v0;
        const bool aligned = ((reinterpret_cast<uintptr_t>(row + v0 * Elem<DT>::kSize) & 15) == 0);
        if (aligned) {
#pragma unroll(kRangeUnroll)
            for (; v + VEC <= v1; v += VEC) {
                float x[VEC];
                unpack<DT>(__ldg(reinterpret_cast<const uint4 *>(row + v * Elem<DT>::kSize)), x);
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    s[e & 3] += (v + e == excl || !kept<DT, F>(x[e], thr)) ? 0.f : ex2(fmaf(x[e], cs, -M));
            }
        }
        return ((s[0] + s[1]) + (s[2] + s[3])) + scalar_sum(*this, v, v1);
    }
    // Masses of the 32 bytes of logits from element v0 (16 bf16 / 8 fp32 tokens) with two
    // 16-byte loads; vec_ok(v0) says whether those loads are aligned.
    static constexpr int kSpan = 32 / Elem<DT>::kSize;
    __device__ __forceinline__ bool vec_ok(int64_t v0) const
    {
        return ((reinterpret_cast<uintptr_t>(row + v0 * Elem<DT>::kSize)) & 15) == 0;
    }
    __device__ __forceinline__ void span(int64_t v0, float (&w)[kSpan]) const
    {
        constexpr int VEC = Elem<DT>::kVec;
        const uint4 *p = reinterpret_cast<const uint4 *>(row + v0 * Elem<DT>::kSize);
        const uint4 a = __ldg(p), b = __ldg(p + 1);
        float x[2 * VEC];
        unpack<DT>(a, x);
        unpack<DT>(b, x + VEC);
#pragma unroll
        for (int e = 0; e < kSpan; ++e)
            w[e] = (v0 + e == excl || !kept<DT, F>(x[e], thr)) ? 0.f : ex2(fmaf(x[e], cs, -M));
    }
};

// Explicit-q residual mass r(v) = max(0, 2^(l_v c - M) / S - q(v)) in probability units.
template <int DT, bool F> struct ResidualMass {
    const char *row;
    const float *qrow;
    float cs, M, inv_s;
    uint32_t thr;  // top-k / top-p cut of the row (0 = none)
    __device__ __forceinline__ float pm(float x) const  // target probability of a logit
    {
        return kept<DT, F>(x, thr) ? ex2(fmaf(x, cs, -M)) * inv_s : 0.f;
    }
    __device__ __forceinline__ float one(int64_t v) const
    {
        return fmaxf(0.f, pm(load1<DT>(row, v)) - __ldg(qrow + v));
    }
    __device__ __forceinline__ float range(int64_t v0, int64_t v1) const
    {
        constexpr int VEC = Elem<DT>::kVec;
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        int64_t v = v0;
        const bool aligned = ((reinterpret_cast<uintptr_t>(row + v0 * Elem<DT>::kSize) & 15) == 0) &&
                             ((reinterpret_cast<uintptr_t>(qrow + v0) & 15) == 0);
        if (aligned) {
#pragma unroll(kRangeUnroll)
            for (; v + VEC <= v1; v += VEC) {
                float x[VEC];
                unpack<DT>(__ldg(reinterpret_cast<const uint4 *>(row + v * Elem<DT>::kSize)), x);
#pragma unroll
                for (int h = 0; h < VEC / 4; ++h) {
                    const float4 q4 = __ldg(reinterpret_cast<const float4 *>(qrow + v) + h);
                    s[0] += fmaxf(0.f, pm(x[4 * h + 0]) - q4.x);
                    s[1] += fmaxf(0.f, pm(x[4 * h + 1]) - q4.y);
                    s[2] += fmaxf(0.f, pm(x[4 * h + 2]) - q4.z);
                    s[3] += fmaxf(0.f, pm(x[4 * h + 3]) - q4.w);
                }
            }
        }
        return ((s[0] + s[1]) + (s[2] + s[3])) + scalar_sum(*this, v, v1);
    }
    static constexpr int kSpan = 32 / Elem<DT>::kSize;
    __device__ __forceinline__ bool vec_ok(int64_t v0) const
    {
        return (((reinterpret_cast<uintptr_t>(row + v0 * Elem<DT>::kSize)) | reinterpret_cast<uintptr_t>(qrow + v0)) &
                15) == 0;
    }
    __device__ __forceinline__ void span(int64_t v0, float (&w)[kSpan]) const
    {
        constexpr int VEC = Elem<DT>::kVec;
        const uint4 *p = reinterpret_cast<const uint4 *>(row + v0 * Elem<DT>::kSize);
        const uint4 a = __ldg(p), b = __ldg(p + 1);
        float x[2 * VEC];
        unpack<DT>(a, x);
        unpack<DT>(b, x + VEC);
        const float4 *q4 = reinterpret_cast<const float4 *>(qrow + v0);
        float qv[kSpan];
#pragma unroll
        for (int h = 0; h < kSpan / 4; ++h) {
            const float4 t = __ldg(q4 + h);
            qv[4 * h + 0] = t.x;
            qv[4 * h + 1] = t.y;
            qv[4 * h + 2] = t.z;
            qv[4 * h + 3] = t.w;
        }
#pragma unroll
        for (int e = 0; e < kSpan; ++e)
            w[e] = fmaxf(0.f, pm(x[e]) - qv[e]);
    }
};

// Smallest v in [lo, hi) whose inclusive prefix mass exceeds theta (masses given by F).
// Three levels: 32 lane segments, 32 sub-segments of the chosen segment, then the
// elements of the chosen sub-segment in order.  When rounding leaves theta beyond the
// range's total, returns the last element with positive mass (or hi - 1).
template <class F>
__device__ int64_t warp_find(const F &f, int64_t lo, int64_t hi, float theta, int lane)
{
    for (int level = 0; level < 2; ++level) {
        const int64_t n = hi - lo;
        if (n <= 32)
            break;
        int64_t seg = (n + 31) / 32;
        if (level == 0)
            seg = (seg + 7) & ~int64_t(7);  // keep segment starts vector aligned
        const int64_t s0 = min(hi, lo + lane * seg), s1 = min(hi, s0 + seg);
        const float tot = f.range(s0, s1);
        const float incl = warp_incl_scan(tot, lane);
        const unsigned hit = __ballot_sync(kFull, incl > theta);
        int L;
        if (hit) {
            L = __ffs(hit) - 1;
        } else {
            const unsigned pos = __ballot_sync(kFull, tot > 0.f);
            if (!pos)
                return hi - 1;
            L = 31 - __clz(pos);
            theta = INFINITY;  // take the last positive element of that segment
        }
        const float excl = __shfl_sync(kFull, incl - tot, L);
        if (theta != INFINITY)
            theta -= excl;
        lo = min(hi, lo + L * seg);
        hi = min(hi, lo + seg);
    }
    // final level: at most 32 elements, one per lane
    const int64_t v = lo + lane;
    const float w = (v < hi) ? f.one(v) : 0.f;
    const float incl = warp_incl_scan(w, lane);
    const unsigned hit = __ballot_sync(kFull, v < hi && incl > theta);
    if (hit)
        return lo + (__ffs(hit) - 1);
    const unsigned pos = __ballot_sync(kFull, w > 0.f);
    return pos ? lo + (31 - __clz(pos)) : hi - 1;
}

// ---- the same search by a whole block (all threads call it; blockDim.x threads, at most 32
// warps).  Thread i owns the kSpan tokens [lo + i * kSpan, ...) of the range (a chunk: at
// most blockDim.x * kSpan tokens), loads them at once (two 16-byte loads of logits), and a
// block scan over the threads' totals finds the thread whose tokens hold theta; that thread
// finishes the search in registers.  One round trip to memory instead of one per level.
struct BlockSearch {
    float wsum[32];
    int hit_thread;
    int pos_thread;
    int64_t token;
};

template <class F>
__device__ __noinline__ int64_t block_find(const F &f, int64_t lo, int64_t hi, float theta, BlockSearch &S)
{
    constexpr int N = F::kSpan;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (int)(blockDim.x >> 5);
    const int64_t s0 = lo + (int64_t)tid * N;
    float w[N];
    if (s0 + N <= hi && f.vec_ok(s0)) {
        f.span(s0, w);
    } else {
#pragma unroll
        for (int e = 0; e < N; ++e)
            w[e] = (s0 + e < hi) ? f.one(s0 + e) : 0.f;
    }
    float tot = 0.f;
#pragma unroll
    for (int e = 0; e < N; ++e)
        tot += w[e];
    float incl = warp_incl_scan(tot, lane);
    if (lane == 31)
        S.wsum[warp] = incl;
    if (tid == 0) {
        S.hit_thread = INT_MAX;
        S.pos_thread = -1;
    }
    __syncthreads();
    float base = 0.f;
    for (int k = 0; k < warp; ++k)
        base += S.wsum[k];
    incl += base;
    const unsigned hit = __ballot_sync(kFull, incl > theta);
    const unsigned pos = __ballot_sync(kFull, tot > 0.f);
    if (lane == 0) {
        if (hit)
            atomicMin(&S.hit_thread, warp * 32 + __ffs(hit) - 1);
        if (pos)
            atomicMax(&S.pos_thread, warp * 32 + 31 - __clz(pos));
    }
    __syncthreads();
    const int h = S.hit_thread;
    if (h != INT_MAX ? tid == h : tid == S.pos_thread) {
        int64_t tok = -1, last = -1;
        float c = incl - tot;
        const float th = h != INT_MAX ? theta : INFINITY;  // rounding left theta beyond the total
#pragma unroll
        for (int e = 0; e < N; ++e) {
            if (w[e] > 0.f)
                last = s0 + e;
            c += w[e];
            if (tok < 0 && c > th)
                tok = s0 + e;
        }
        S.token = tok >= 0 ? tok : (last >= 0 ? last : hi - 1);
    }
    if (h == INT_MAX && S.pos_thread < 0 && tid == 0)
        S.token = hi - 1;
    __syncthreads();
    const int64_t tok = S.token;
    __syncthreads();  // S is reused by the caller's next search
    (void)nw;
    return tok;
}

// Total mass of [lo, hi) by a whole block (thread i: kSpan tokens from lo + i * kSpan).
template <class F> __device__ __noinline__ float block_range_mass(const F &f, int64_t lo, int64_t hi, BlockSearch &S)
{
    constexpr int N = F::kSpan;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = (int)(blockDim.x >> 5);
    float tot = 0.f;
    for (int64_t s0 = lo + (int64_t)tid * N; s0 < hi; s0 += (int64_t)blockDim.x * N) {
        float w[N];
        if (s0 + N <= hi && f.vec_ok(s0)) {
            f.span(s0, w);
        } else {
#pragma unroll
            for (int e = 0; e < N; ++e)
                w[e] = (s0 + e < hi) ? f.one(s0 + e) : 0.f;
        }
#pragma unroll
        for (int e = 0; e < N; ++e)
            tot += w[e];
    }
    tot = warp_sum(tot);
    if (lane == 0)
        S.wsum[warp] = tot;
    __syncthreads();
    float z = 0.f;
    for (int k = 0; k < nw; ++k)
        z += S.wsum[k];
    __syncthreads();
    return z;
}

// Masses of the chunks of row t relative to 2^M (K1 partials), one chunk optionally
// replaced by a mass computed separately (the chunk of x* without x*).
struct ChunkMassFromPartials {
    const float2 *pp;
    float cs, M;
    int override_chunk;
    float override_mass;
    __device__ __forceinline__ float operator()(int c) const
    {
        if (c == override_chunk)
            return override_mass;
        const float2 pc = pp[c];
        return (pc.x == -INFINITY) ? 0.f : pc.y * ex2(pc.x * cs - M);
    }
};

// Total mass of [lo, hi) by the warp: 32 contiguous, vector-aligned segments, one per lane.
template <class F> __device__ __forceinline__ float warp_range_mass(const F &f, int64_t lo, int64_t hi, int lane)
{
    const int64_t seg = (((hi - lo + 31) / 32) + 7) & ~int64_t(7);
    const int64_t s0 = min(hi, lo + lane * seg), s1 = min(hi, s0 + seg);
    return warp_sum(f.range(s0, s1));
}



// Warp scan over the chunk masses: total Z, then the chunk holding u * Z and the
// remaining threshold inside it.  Both passes use the same scan, so they agree bit for bit.
template <class CM>
__device__ __forceinline__ float chunk_total(const CM &cm, int nchunks, int lane)
{
    float carry = 0.f;
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
        const float m = (c0 + lane < nchunks) ? cm(c0 + lane) : 0.f;
        const float incl = warp_incl_scan(m, lane);
        carry += __shfl_sync(kFull, incl, 31);
    }
    return carry;
}

template <class CM>
__device__ __forceinline__ int chunk_locate(const CM &cm, int nchunks, float theta, int lane, float &theta_in)
{
    float carry = 0.f;
    int last_pos = -1;
    float last_mass = 0.f;
    for (int c0 = 0; c0 < nchunks; c0 += 32) {
        const float m = (c0 + lane < nchunks) ? cm(c0 + lane) : 0.f;
        const float incl = warp_incl_scan(m, lane) + carry;
        const unsigned hit = __ballot_sync(kFull, incl > theta);
        if (hit) {
            const int L = __ffs(hit) - 1;
            theta_in = theta - __shfl_sync(kFull, incl - m, L);
            return c0 + L;
        }
        const unsigned pos = __ballot_sync(kFull, m > 0.f);
        if (pos) {
            const int L = 31 - __clz(pos);
            last_pos = c0 + L;
            last_mass = __shfl_sync(kFull, m, L);
        }
        carry = __shfl_sync(kFull, incl, 31);
    }
    // rounding left theta at or beyond the total: last chunk with mass, its last element
    theta_in = INFINITY;
    (void)last_mass;
    return last_pos < 0 ? nchunks - 1 : last_pos;
}

// Residual mass sum max(0, p(v) - q(v)) over the chunk [lo, hi) by one warp: lane-strided
// 16-byte groups of target logits and draft probabilities, four groups in flight per lane.
template <int DT, bool F, int U = 4, bool STAGE = false>
__device__ __forceinline__ float warp_residual_chunk(const ResidualMass<DT, F> &f, int64_t lo, int64_t hi, int lane,
                                                     float *qdst = nullptr)
{
    constexpr int VEC = Elem<DT>::kVec;
    constexpr int ES = Elem<DT>::kSize;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int64_t tail = lo;
    if (STAGE && DT == 1 && (((reinterpret_cast<uintptr_t>(f.row + lo * ES) | reinterpret_cast<uintptr_t>(f.qrow + lo) |
                               reinterpret_cast<uintptr_t>(qdst + lo)) & 15) == 0)) {
        // bf16 rows with q in host memory.  Lane l sums the 8 tokens of group g = g0 + l as the
        // plain path below does (the same order, so the same sums), but q is loaded as two
        // contiguous 512-byte spans per 256 tokens (q[4l..4l+3] and q[128+4l..]) and handed to
        // the lanes that need it by shuffles: a 16-byte load per lane at a 32-byte stride would
        // make each load instruction fetch every line of a 1 KB span over the host link, and the
        // two instructions fetch them twice.  U groups are loaded before any copy is stored: a
        // store might alias a later load as far as the compiler knows.
        const int64_t ng = (hi - lo) / VEC;
        const int64_t nfull = ng / 32;  // whole 256-token spans
        const int src0 = (2 * lane) & 31, src1 = (2 * lane + 1) & 31;
        const bool lo_half = lane < 16;
        for (int64_t s0 = 0; s0 < nfull; s0 += U) {
            uint4 rw[U], qa[U], qb[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (s0 + u < nfull) {
                    const int64_t base = lo + (s0 + u) * 256;
                    rw[u] = ld_stream(f.row + (base + 8 * lane) * ES);
                    qa[u] = ld_stream(f.qrow + base + 4 * lane);
                    qb[u] = ld_stream(f.qrow + base + 128 + 4 * lane);
                }
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (s0 + u < nfull) {
                    const int64_t base = lo + (s0 + u) * 256;
                    *reinterpret_cast<uint4 *>(qdst + base + 4 * lane) = qa[u];
                    *reinterpret_cast<uint4 *>(qdst + base + 128 + 4 * lane) = qb[u];
                    auto pick = [&](uint32_t a, uint32_t b, int src) {
                        const uint32_t x = __shfl_sync(kFull, a, src), y = __shfl_sync(kFull, b, src);
                        return __uint_as_float(lo_half ? x : y);
                    };
                    const float q8[8] = {pick(qa[u].x, qb[u].x, src0), pick(qa[u].y, qb[u].y, src0),
                                         pick(qa[u].z, qb[u].z, src0), pick(qa[u].w, qb[u].w, src0),
                                         pick(qa[u].x, qb[u].x, src1), pick(qa[u].y, qb[u].y, src1),
                                         pick(qa[u].z, qb[u].z, src1), pick(qa[u].w, qb[u].w, src1)};
                    float x[VEC];
                    unpack<DT>(rw[u], x);
#pragma unroll
                    for (int h = 0; h < VEC / 4; ++h) {
                        acc[0] += fmaxf(0.f, f.pm(x[4 * h + 0]) - q8[4 * h + 0]);
                        acc[1] += fmaxf(0.f, f.pm(x[4 * h + 1]) - q8[4 * h + 1]);
                        acc[2] += fmaxf(0.f, f.pm(x[4 * h + 2]) - q8[4 * h + 2]);
                        acc[3] += fmaxf(0.f, f.pm(x[4 * h + 3]) - q8[4 * h + 3]);
                    }
                }
        }
        // the groups past the last whole span, as the plain path
        for (int64_t g = nfull * 32 + lane; g < ng; g += 32) {
            const int64_t v = lo + g * VEC;
            float x[VEC];
            unpack<DT>(ld_stream(f.row + v * ES), x);
#pragma unroll
            for (int h = 0; h < VEC / 4; ++h) {
                const uint4 qw = ld_stream(f.qrow + v + 4 * h);
                *reinterpret_cast<uint4 *>(qdst + v + 4 * h) = qw;
                acc[0] += fmaxf(0.f, f.pm(x[4 * h + 0]) - __uint_as_float(qw.x));
                acc[1] += fmaxf(0.f, f.pm(x[4 * h + 1]) - __uint_as_float(qw.y));
                acc[2] += fmaxf(0.f, f.pm(x[4 * h + 2]) - __uint_as_float(qw.z));
                acc[3] += fmaxf(0.f, f.pm(x[4 * h + 3]) - __uint_as_float(qw.w));
            }
        }
        tail = lo + ng * VEC;
    } else if (STAGE && ((reinterpret_cast<uintptr_t>(f.row + lo * ES) | reinterpret_cast<uintptr_t>(f.qrow + lo) |
                          reinterpret_cast<uintptr_t>(qdst + lo)) & 15) == 0) {
        // U groups loaded before any is stored (see above); fp32 q loads are contiguous per warp
        const int64_t ng = (hi - lo) / VEC;
        for (int64_t g0 = lane; g0 < ng; g0 += 32 * U) {
            uint4 rw[U], qw[U][VEC / 4];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t g = g0 + 32 * u;
                if (g < ng) {
                    const int64_t v = lo + g * VEC;
                    rw[u] = ld_stream(f.row + v * ES);
#pragma unroll
                    for (int h = 0; h < VEC / 4; ++h)
                        qw[u][h] = ld_stream(f.qrow + v + 4 * h);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t g = g0 + 32 * u;
                if (g < ng) {
                    const int64_t v = lo + g * VEC;
                    float x[VEC];
                    unpack<DT>(rw[u], x);
#pragma unroll
                    for (int h = 0; h < VEC / 4; ++h) {
                        *reinterpret_cast<uint4 *>(qdst + v + 4 * h) = qw[u][h];
                        acc[0] += fmaxf(0.f, f.pm(x[4 * h + 0]) - __uint_as_float(qw[u][h].x));
                        acc[1] += fmaxf(0.f, f.pm(x[4 * h + 1]) - __uint_as_float(qw[u][h].y));
                        acc[2] += fmaxf(0.f, f.pm(x[4 * h + 2]) - __uint_as_float(qw[u][h].z));
                        acc[3] += fmaxf(0.f, f.pm(x[4 * h + 3]) - __uint_as_float(qw[u][h].w));
                    }
                }
            }
        }
        tail = lo + ng * VEC;
    } else if (((reinterpret_cast<uintptr_t>(f.row + lo * ES) | reinterpret_cast<uintptr_t>(f.qrow + lo)) & 15) == 0) {
        const int64_t ng = (hi - lo) / VEC;
#pragma unroll(U)
        for (int64_t g = lane; g < ng; g += 32) {
            const int64_t v = lo + g * VEC;
            float x[VEC];
            unpack<DT>(ld_stream(f.row + v * ES), x);
#pragma unroll
            for (int h = 0; h < VEC / 4; ++h) {
                const uint4 qw = ld_stream(f.qrow + v + 4 * h);
                if (STAGE)  // the device copy of the draft row, for the draw that follows
                    *reinterpret_cast<uint4 *>(qdst + v + 4 * h) = qw;
                acc[0] += fmaxf(0.f, f.pm(x[4 * h + 0]) - __uint_as_float(qw.x));
                acc[1] += fmaxf(0.f, f.pm(x[4 * h + 1]) - __uint_as_float(qw.y));
                acc[2] += fmaxf(0.f, f.pm(x[4 * h + 2]) - __uint_as_float(qw.z));
                acc[3] += fmaxf(0.f, f.pm(x[4 * h + 3]) - __uint_as_float(qw.w));
            }
        }
        tail = lo + ng * VEC;
    }
    for (int64_t v = tail + lane; v < hi; v += 32) {
        acc[0] += f.one(v);
        if (STAGE)
            qdst[v] = __ldg(f.qrow + v);
    }
    return warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
}


struct ChunkMassFromL2 {  // masses written by other warps of this launch: read past L1
    const float *z;
    __device__ __forceinline__ float operator()(int c) const { return __ldcg(z + c); }
};


}  // namespace
}  // namespace specrej
