// spec_reject.cu -- batched verify-side rejection sampler for speculative decoding,
// hand-written for GB300 (sm_103a).  Implements the C ABI of include/spec_reject.h.
//
// The method (speculative sampling, "第12章 投机解码：以小博大" §12.2.1-§12.2.4, §12.3.2):
// per request, accept draft x* with probability min(1, p/q) in order, stop at the first
// rejection, draw the recovered token from max(0, p - q) there (one-hot q: p without x*,
// §12.9), or the bonus token from p after the last draft; at temperature 0 compare with
// the argmax instead.
//
// Structure on the GPU (every step is a kernel of this library; nothing runs on the host).
// Rows are split into chunks of 8 KB of logits (4096 bf16 / 2048 fp32); a chunk reduces to a
// partial: sampling rows (m_c, s_c) with m_c the chunk max and s_c = sum 2^(l c - fl(m_c c)),
// c = log2(e) / T_r; greedy rows (max, lowest index of the max).
//
//   KL  lazy_kernel, the first-rejection pass: every call without diagnostics whose rows are
//       16-byte aligned (top-k / top-p: bf16 rows and at least 64 requests; rows in pinned
//       host memory: at least 64 requests).  After a one-block layout check (lazy_init_kernel,
//       chained by programmatic dependent launch), persistent blocks take requests from an
//       atomic queue.  Per request the block streams rows t_0, t_1, ... through warp-private
//       TMA rings (cp.async.bulk into shared memory, bounded mbarrier waits), reduces each
//       chunk to its partial in shared memory, and warp 0 combines the row and decides
//       position i; the walk stops at the first rejection j.  An explicit-q rejection runs the
//       residual pass over target row t_j and draft row j (chunk masses of max(0, p - q), all
//       warps); the whole block then draws the output token (chunk scan, then block_find over
//       the located chunk) and warp 0 writes the outputs.  Batches too small to fill the GPU
//       one block per request run with thread-block clusters of 2, 4 or 8 blocks per request
//       (chunks spread over every warp of the cluster, partials gathered in the leader block
//       through distributed shared memory).  The last requests of a large batch run in a
//       second launch, two blocks each, chained to the first.  With cuts, each reached row is
//       cut in the block (kl_cut_row: counts over a window of the largest keys, marked with
//       packed compares), and the output row's residual and draw read only its listed kept
//       tokens when they are few (kl_list_draw); batches of at most 4 requests per SM take a
//       16-warp build of this kernel (spec_reject_cut16.cu compiles this file again).  With
//       rows in host memory, rows are read over the host link with 16-byte loads and copied to
//       the device for the residual pass and the draw.
//   K1  rowstats_wr_kernel / rowstats_kernel, the full pass's row statistics: every chunk of
//       every row, warp-private TMA rings (register-staged 16-byte loads for misaligned rows);
//       block 0 checks the layout.
//   K1F filter_kernel: top-k / top-p cut of each filtered row by one thread-block cluster.
//   K2  finalize_kernel: one warp per request; combines the chunk partials of each verify row,
//       takes the acceptance decisions (ballot for the first rejection) and draws the bonus /
//       one-hot recoveries (chunk scan + three-level warp descent).
//   K3  residual_kernel: explicit-q recoveries; warps stream (request, chunk) units of target
//       row j and draft row j; the warp completing a request's last chunk draws.
//   Also: metrics_kernel (acceptance counters), tree_walk_kernel (greedy tree verification),
//   ngram_kernel (n-gram proposer), the diagnostic kernels and the host-row staging kernel.
//
// Every reduction has a fixed order (warp butterflies, sequential chunk combines), so
// identical inputs give identical outputs; there are no floating-point atomics.  No block
// waits for another block except through a thread-block cluster's hardware barrier, which
// every block of the cluster takes in the same order; every mbarrier wait is bounded.

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <limits.h>
#include <math.h>

#include <mutex>

#include "spec_reject.h"
#include "common.cuh"

namespace specrej {
namespace {

// Programmatic dependent launch: a kernel launched as the dependent of the one before it on the
// stream may be scheduled while that one still runs (once all its blocks have started and
// allowed it); it waits here for that kernel's completion and writes before reading anything.
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void wait_for_prerequisite() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
template <int DT>
__global__ void __launch_bounds__(kThreads, SPEC_LDG_MIN_BLOCKS) rowstats_kernel(Params P, int force_argmax)
{
    allow_dependents();  // the next kernel of the full pass may take SM slots as these blocks finish
    if (blockIdx.x == 0 && force_argmax != kArgmaxKeepErrors)
        validate_layout(P);
    if (P.B == 0)
        return;
    const int lane = threadIdx.x & 31;
    const int64_t nunits = P.T * (int64_t)P.nchunks;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t per = (nunits + nw - 1) / nw;
    const int64_t u0 = gw * per;
    const int64_t u1 = min(nunits, u0 + per);
    RowInfo ri;
    for (int64_t u = u0; u < u1; ++u) {
        const int64_t t = u / P.nchunks;
        const int c = (int)(u - t * P.nchunks);
        if (t != ri.t)
            row_info(P, t, force_argmax, ri);
        rowstats_unit<DT>(P, t, c, ri.greedy, ri.cs, lane);
    }
}

// ---------------------------------------------------------------------------------------
// K1 with warp-private TMA pipelines
// ---------------------------------------------------------------------------------------
//
// Each warp streams its own contiguous range of units through its own ring of kWrStages
// shared-memory slots: lane 0 keeps kWrStages bulk copies in flight ahead of the warp, the
// warp copies a landed unit into registers, lane 0 immediately reuses the slot for the unit
// kWrStages further on, and the warp reduces the unit from registers.  No warp ever waits
// for another, and a slot's mbarrier is only waited on by the warp that refills it, one
// phase at a time, so every parity wait is unambiguous.

#ifndef SPEC_WR_WARPS
#define SPEC_WR_WARPS 4       // warps per block
#endif
#ifndef SPEC_WR_STAGES
#define SPEC_WR_STAGES 3      // slots per warp
#endif
#ifndef SPEC_WR_MIN_BLOCKS
#define SPEC_WR_MIN_BLOCKS 2  // 2 blocks x 4 warps x 3 slots x 8 KB = 192 KB of logits in flight per SM
#endif
constexpr int kWrWarps = SPEC_WR_WARPS;
constexpr int kWrStages = SPEC_WR_STAGES;
constexpr int kWrThreads = kWrWarps * 32;

template <int DT>
__global__ void __launch_bounds__(kWrThreads, SPEC_WR_MIN_BLOCKS) rowstats_wr_kernel(Params P, int force_argmax)
{
    allow_dependents();  // the next kernel of the full pass may take SM slots as these blocks finish
    constexpr int VEC = Elem<DT>::kVec;
    constexpr int ES = Elem<DT>::kSize;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kWrWarps * kWrStages];

    if (blockIdx.x == 0 && force_argmax != kArgmaxKeepErrors)
        validate_layout(P);
    if (P.B == 0)
        return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x < kWrWarps * kWrStages)
        mbar_init(&full[threadIdx.x], 1);
    mbar_fence_init();
    __syncthreads();

    const int64_t nunits = P.T * (int64_t)P.nchunks;
    const int64_t nw = (int64_t)gridDim.x * kWrWarps;
    const int64_t per = (nunits + nw - 1) / nw;
    const int64_t u0 = ((int64_t)blockIdx.x * kWrWarps + warp) * per;
    const int64_t n = max((int64_t)0, min(nunits, u0 + per) - u0);
    unsigned char *slots = ring + (size_t)warp * kWrStages * kUnitBytes;
    uint64_t *bars = full + warp * kWrStages;

    // issue side (lane 0): unit u0 + qi, walked incrementally
    int64_t it = u0 / P.nchunks;
    int ic = (int)(u0 - it * P.nchunks);
    int64_t qi = 0;
    auto issue = [&]() {
        const int s = (int)(qi % kWrStages);
        const int64_t lo = (int64_t)ic * P.chunk;
        const int64_t hi = min((int64_t)P.V, lo + P.chunk);
        const uint32_t bytes = (uint32_t)((hi - lo) * ES) & ~15u;
        mbar_arrive_expect_tx(&bars[s], bytes);
        if (bytes)
            bulk_g2s(slots + (size_t)s * kUnitBytes, row_ptr<DT>(P, it) + lo * ES, bytes, &bars[s]);
        ++qi;
        if (++ic == P.nchunks) {
            ic = 0;
            ++it;
        }
    };
    if (lane == 0)
        while (qi < n && qi < kWrStages)
            issue();

    // compute side: unit u0 + q, row and request walked incrementally
    int64_t t = u0 / P.nchunks;
    int c = (int)(u0 - t * P.nchunks);
    int r = n > 0 ? find_request(P, t) : 0;
    int64_t r_end = (int64_t)__ldg(P.cu + r + 1) + r + 1;
    int64_t info_t = -1;
    bool greedy = true;
    float cs = 0.f;
    int64_t q = 0;
    for (; q < n; ++q) {
        const int s = (int)(q % kWrStages);
        if (!__all_sync(kFull, mbar_wait(&bars[s], (uint32_t)(q / kWrStages) & 1, P.err)))
            break;
        UnitRange R;
        R.lo = (int64_t)c * P.chunk;
        R.hi = min((int64_t)P.V, R.lo + P.chunk);
        R.vlo = R.lo;
        R.nvec = ((R.hi - R.lo) * ES) / 16;
        R.vhi = R.vlo + R.nvec * VEC;
        const uint4 *stage = reinterpret_cast<const uint4 *>(slots + (size_t)s * kUnitBytes);
        uint4 v[kVecPerLane];
#pragma unroll
        for (int k = 0; k < kVecPerLane; ++k) {
            const int vi = k * 32 + lane;
            v[k] = (vi < R.nvec) ? stage[vi] : neg_inf_vec<DT>();
        }
        __syncwarp();
        if (lane == 0 && qi < n)
            issue();  // the slot is in registers: refill it with the unit kWrStages ahead
        if (t != info_t) {
            info_t = t;
            while (t >= r_end && r < P.B - 1) {
                ++r;
                r_end = (int64_t)__ldg(P.cu + r + 1) + r + 1;
            }
            const float temp = __ldg(P.temp + r);
            greedy = force_argmax || !(temp > 0.f);
            cs = greedy ? 0.f : kLog2e / temp;
        }
        const char *row = row_ptr<DT>(P, t);
        if (greedy)
            argmax_regs<DT>(P.part + t * P.nchunks + c, lane, v, R, row);
        else
            softmax_regs<DT>(P.part + t * P.nchunks + c, cs, lane, v, R, row);
        if (++c == P.nchunks) {
            c = 0;
            ++t;
        }
    }
    // gave up on a wait: let this warp's copies still in flight land before exiting
    if (lane == 0)
        for (int64_t q2 = q + 1; q2 < qi; ++q2)
            mbar_wait(&bars[q2 % kWrStages], (uint32_t)(q2 / kWrStages) & 1, P.err);
}

// ---------------------------------------------------------------------------------------
// K1F: top-k / top-p cut of a target row, one thread-block cluster per row
// ---------------------------------------------------------------------------------------
//
// The cluster holds the whole row in distributed shared memory (each block a slice of whole
// chunks, brought in with one bulk copy).  K1 has already written the row's unfiltered chunk
// partials, which give the row maximum m, each chunk's maximum and (for top-p alone) the
// normaliser Z.  A token's mass is 2^(l c - m c) in fixed point (2^-32 units), so the sums
// that decide the cut are integer sums and no decision depends on scheduling.
//
// bf16 rows first try one pass: each warp counts its chunk's tokens by their order key's
// offset below the maximum's key, over the kFKeys largest keys.  One count and one mass per
// key give the exact k-th largest key, S_k, the exact top-p key, and each chunk's partial
// (m_c, s_c) over the survivors, with no second pass.  A cut further down than kFKeys keys,
// and every fp32 row, takes the general path:
//   1. one pass: token counts over kFBins bins of d = m c - l c (kFBinScale bins per unit of
//      log2 relative probability, the last bin open-ended).  The bin is a monotone function of
//      the logit, so every token of a lower bin outranks every token of a higher one.
//   2. the last bin that can hold a survivor: top-k, the bin where the count scan reaches k;
//      top-p alone, the bin where a lower bound of the cumulative mass (each bin's count times
//      the least mass its tokens can have) reaches top_p * Z.
//   3. one pass: every token up to that bin goes into a candidate list (order key, position).
//   4. from the list: the k-th largest key (ranking the tokens of its bin), S_k = the exact
//      mass at or above it, the bin where the exact cumulative mass reaches top_p * S_k and
//      the exact key inside it, and each chunk's partial over the survivors.
// A list longer than kFList falls back to passes over the slice (mass histograms and radix
// selects on the order key), and a bin with more than kFWindow tokens is resolved by a radix
// select over the slice.  The row's cut key goes to K2 / K3.  Every block of a cluster takes
// every cluster barrier, in the same order, and makes the same decisions from the same
// cluster-wide totals.

namespace cg = cooperative_groups;

constexpr int kFilterThreads = 512;
constexpr int kFilterWarps = kFilterThreads / 32;
constexpr int kFilterMaxChunksPerBlock = 20;  // 20 x 8 KB = 160 KB of the row per block
constexpr int kFilterMaxCluster = 8;
constexpr int kFBins = 2048;                  // bins of d
constexpr float kFBinScale = 64.f;            // bins per unit of log2 relative probability
constexpr int kFList = 2048;                  // candidate list entries (per block, and merged)
constexpr int kFWindow = 512;                 // tokens of one bin ranked directly
#ifndef SPEC_FILTER_KEYS
#define SPEC_FILTER_KEYS 512
#endif
#ifndef SPEC_FILTER_LOADS
#define SPEC_FILTER_LOADS 4  // 16-byte loads in flight per lane in the one-pass count
#endif
constexpr int kFKeys = SPEC_FILTER_KEYS;      // bf16 one-pass window: the largest keys counted
static_assert(kFBins == 4 * kFilterThreads, "bins are owned four per thread");
static_assert(kFWindow <= kFilterThreads, "one window token per thread");

// This block's part of a target row, read in place (global memory).
struct RowSlice {
    const char *p;  // element 0 of the part
    bool vec;       // 16-byte aligned: 16-byte loads
};

// fn(x, i) for every element i of the part's [e0, e1) with threads tid0, tid0 + step, ...:
// 16-byte vectors over the aligned middle (e0 a multiple of the vector width), then the
// scalar tail; scalar loads throughout when the part is not 16-byte aligned.
template <int DT, class Fn>
__device__ __forceinline__ void slice_range(const RowSlice &sl, int64_t e0, int64_t e1, int tid0, int step, Fn fn)
{
    constexpr int VEC = Elem<DT>::kVec;
    int tail0 = (int)e0;
    if (sl.vec) {
        const int v0 = (int)(e0 / VEC), v1 = (int)(e1 / VEC);
        for (int v = v0 + tid0; v < v1; v += step) {
            float x[VEC];
            unpack<DT>(ld_stream(sl.p + (size_t)v * 16), x);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                fn(x[e], v * VEC + e);
        }
        tail0 = v1 * VEC;
    }
    for (int i = tail0 + tid0; i < (int)e1; i += step)
        fn(load1<DT>(sl.p, i), i);
}

template <int DT, class Fn> __device__ __forceinline__ void slice_for_each(const RowSlice &sl, int64_t n, Fn fn)
{
    slice_range<DT>(sl, 0, n, threadIdx.x, blockDim.x, fn);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum_f64(double v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Scalars of one K1F block.
struct FilterShared {
    unsigned long long red[kFilterWarps];
    double z;
    float maxv;
    float cmax[kFilterMaxChunksPerBlock];  // K1's maxima of this block's chunks
    unsigned nlocal;
    int nlist;
    int pos;
    unsigned long long above;
    unsigned long long sum;
    unsigned best;
    unsigned nwin;
};

// Arrays of the general path.
struct FilterGeneral {
    unsigned cnt[kFBins];                // bin counts (cluster totals after the sum)
    unsigned long long mh[kFBins];       // bin masses: 64-bit sums, or (list path) 16-bit halves
    unsigned long long local[kFList];    // this block's candidates; after the merge, scratch
    unsigned long long list[kFList];     // the cluster's candidates: key << 32 | position
};

// Arrays of the bf16 one-pass path.
struct FilterKeys {
    unsigned hc[kFilterMaxChunksPerBlock][kFKeys + 32];  // per chunk: tokens per key offset, then
                                                         // one sink per lane for the rest
    unsigned bh[kFKeys];                                 // per key offset: block, then cluster totals
    unsigned gather[kFilterMaxCluster][kFKeys];          // every block's totals, pushed by its owner
    unsigned long long km[kFKeys];                       // mass of one token at each key offset
};

union FilterArrays {
    FilterGeneral g;
    FilterKeys k;
};

// Sum over the block (every thread gets it).
__device__ __forceinline__ unsigned long long block_sum_u64(FilterShared &S, unsigned long long v)
{
    v = warp_sum_u64(v);
    __syncthreads();  // S.red is free
    if ((threadIdx.x & 31) == 0)
        S.red[threadIdx.x >> 5] = v;
    __syncthreads();
    unsigned long long t = 0;
    for (int w = 0; w < kFilterWarps; ++w)
        t += S.red[w];
    return t;
}

// Sum of a per-thread value over the block, then over the cluster (every thread gets it).
__device__ __forceinline__ unsigned long long cluster_sum_u64(FilterShared &S, cg::cluster_group &cluster, int csize,
                                                              unsigned long long v)
{
    const unsigned long long b = block_sum_u64(S, v);
    if (threadIdx.x == 0)
        S.sum = b;
    cluster.sync();
    unsigned long long t = 0;
    for (int q = 0; q < csize; ++q)
        t += *cluster.map_shared_rank(&S.sum, q);
    cluster.sync();  // every block has read every S.sum before any is rewritten
    return t;
}

// In-place cluster-wide sum of the first nb entries of every block's histogram h (h at the
// same offset in every block).  Threads own nb / blockDim consecutive bins (nb <= 4 *
// blockDim, a multiple of blockDim or at most blockDim).
template <class W>
__device__ __forceinline__ void cluster_sum_hist(W *h, cg::cluster_group &cluster, int csize, int nb)
{
    const int per = nb > (int)blockDim.x ? nb / (int)blockDim.x : 1;
    const int b0 = threadIdx.x * per;
    W v[4] = {0, 0, 0, 0};
    cluster.sync();  // every block's histogram is complete
    if (b0 < nb)
        for (int q = 0; q < csize; ++q) {
            const W *hq = cluster.map_shared_rank(h, q);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (k < per)
                    v[k] += hq[b0 + k];
        }
    cluster.sync();  // every block has read every histogram
    if (b0 < nb)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < per)
                h[b0 + k] = v[k];
    __syncthreads();
}

// Scan of weights w(0..nb) in order: the first position i at which
// above0 + w(0) + ... + w(i) >= target.  Leaves i in S.pos (-1 when the total falls short)
// and above0 + w(0) + ... + w(i - 1) in S.above.  Same ownership as cluster_sum_hist.
template <class WF>
__device__ __forceinline__ void find_crossing(FilterShared &S, int nb, unsigned long long above0,
                                              unsigned long long target, WF w)
{
    const int per = nb > (int)blockDim.x ? nb / (int)blockDim.x : 1;
    const int b0 = threadIdx.x * per;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long mine = 0;
    if (b0 < nb)
        for (int k = 0; k < per; ++k)
            mine += w(b0 + k);
    unsigned long long inc = mine;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o)
            inc += y;
    }
    __syncthreads();  // S.red and S.pos are free
    if (threadIdx.x == 0)
        S.pos = -1;
    if (lane == 31)
        S.red[warp] = inc;
    __syncthreads();
    // exclusive prefix of the warp totals, by a shuffle scan over lanes < number of warps
    unsigned long long wt = lane < (int)(blockDim.x >> 5) ? S.red[lane] : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(kFull, wt, o);
        if (lane >= o)
            wt += y;
    }
    const unsigned long long before = warp > 0 ? __shfl_sync(kFull, wt, warp - 1) : 0ull;
    unsigned long long c = above0 + before + inc - mine;
    if (b0 < nb && c < target && c + mine >= target)
        for (int k = 0; k < per; ++k) {
            const unsigned long long wk = w(b0 + k);
            if (c + wk >= target) {
                S.pos = b0 + k;
                S.above = c;
                break;
            }
            c += wk;
        }
    __syncthreads();
}

template <int DT>
__global__ void __launch_bounds__(kFilterThreads, 2) filter_kernel(Params P, int csize)
{
    allow_dependents();
    wait_for_prerequisite();  // the row statistics
    constexpr int KEY_BITS = DT ? 16 : 32;
    constexpr int ES = Elem<DT>::kSize;
    __shared__ FilterShared S;
    __shared__ FilterArrays U;

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int64_t t = blockIdx.x / csize;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (t >= P.T || P.B == 0)
        return;  // uniform over the cluster
    const int r = find_request(P, t);
    const float temp = P.temp[r];
    const int32_t tk = P.top_k ? P.top_k[r] : 0;
    const float tp = P.top_p ? P.top_p[r] : 1.f;
    const bool use_k = tk > 0 && tk < P.V;
    const bool use_p = tp > 0.f && tp < 1.f;
    if (!(temp > 0.f) || !(use_k || use_p)) {
        if (rank == 0 && threadIdx.x == 0)
            P.thr[t] = 0;
        return;  // uniform over the cluster
    }
    const float cs = kLog2e / temp;
    const int cpc = (P.nchunks + csize - 1) / csize;
    const int c0 = min(P.nchunks, rank * cpc), c1 = min(P.nchunks, c0 + cpc);
    const int64_t lo = (int64_t)c0 * P.chunk;
    const int64_t n = max((int64_t)0, min((int64_t)P.V, (int64_t)c1 * P.chunk) - lo);
    const char *row = row_ptr<DT>(P, t);
    float2 *pp = P.part + t * P.nchunks;

    // ---- 0. m (and Z) from K1's partials; the row itself is read in place
    const RowSlice slice{row + lo * ES, (reinterpret_cast<uintptr_t>(row + lo * ES) & 15) == 0};
    if (warp == 0) {
        float mm = -INFINITY;
        for (int c = lane; c < P.nchunks; c += 32)
            mm = fmaxf(mm, pp[c].x);
        mm = warp_max(mm);
        double z = 0.0;
        if (!use_k && mm > -INFINITY) {
            const float Mm = mm * cs;
            for (int c = lane; c < P.nchunks; c += 32) {
                const float2 pc = pp[c];
                if (pc.x != -INFINITY)
                    z += (double)pc.y * (double)ex2(pc.x * cs - Mm);
            }
            z = warp_sum_f64(z);
        }
        if (lane == 0) {
            S.maxv = mm;
            S.z = z * 4294967296.0;
        }
        if (lane < c1 - c0)
            S.cmax[lane] = pp[c0 + lane].x;
    }
    __syncthreads();
    const float m = S.maxv;
    if (!(m > -INFINITY)) {  // no finite logit in the row (the same in every block): no cut
        if (rank == 0 && threadIdx.x == 0)
            P.thr[t] = 0;
        return;
    }
    const float M = m * cs;
    auto fx = [&](float x) -> unsigned long long {  // mass 2^(x c - M) in units of 2^-32
        return __float2ull_rn(ex2(fmaf(x, cs, -M)) * 4294967296.0f);
    };
    // s_c of K1's format from a fixed-point sum 2^32 * sum 2^(x c - Mc)
    auto fx_chunk = [&](float x, float Mc) -> unsigned long long {
        return __float2ull_rn(ex2(fmaf(x, cs, -Mc)) * 4294967296.0f);
    };
    constexpr float kTwoM32 = 2.3283064365386963e-10f;  // 2^-32

    uint32_t thr = 0;
    bool done = false;

    // ---- bf16: one pass over the kFKeys largest keys
    if constexpr (DT == 1) {
        const int nck = c1 - c0;
        const uint32_t kmax = key_of<1>(m);
        for (int i = threadIdx.x; i < nck * (kFKeys + 32); i += blockDim.x)
            (&U.k.hc[0][0])[i] = 0u;
        __syncthreads();
        // When the window holds no negative logit, a token's offset is kmax - 0x8000 minus its raw
        // bits (negative logits wrap far above the window); otherwise the full order key.
        const bool plain = kmax >= 0x8000u + (uint32_t)kFKeys;
        for (int ci = warp; ci < nck; ci += kFilterWarps) {
            unsigned *h = U.k.hc[ci];
            const uint32_t sink = (uint32_t)kFKeys + (uint32_t)lane;
            const int e0 = ci * P.chunk, e1 = min((int)n, e0 + P.chunk);
            // no branch: offsets outside the window land in this lane's own sink
            auto count = [&](uint32_t b16) {  // bf16 bits in the low half
                uint32_t off;
                if (plain) {
                    off = kmax - 0x8000u - b16;
                } else {
                    const uint32_t sg = (uint32_t)((int32_t)(b16 << 16) >> 31);
                    off = kmax - (0x8000u + (((b16 & 0x7fffu) ^ sg) - sg));
                }
                atomicAdd(&h[min(off, sink)], 1u);
            };
            auto count8 = [&](const uint4 &w) {
                count(w.x & 0xffffu);
                count(w.x >> 16);
                count(w.y & 0xffffu);
                count(w.y >> 16);
                count(w.z & 0xffffu);
                count(w.z >> 16);
                count(w.w & 0xffffu);
                count(w.w >> 16);
            };
            int tail0 = e0;
            if (slice.vec) {
                constexpr int NL = SPEC_FILTER_LOADS;
                const int v1 = e1 / 8;
                for (int v = e0 / 8 + lane; v < v1; v += NL * 32) {  // NL 16-byte loads in flight
                    uint4 w[NL];
#pragma unroll
                    for (int u = 0; u < NL; ++u)
                        if (v + 32 * u < v1)
                            w[u] = ld_stream(slice.p + (size_t)(v + 32 * u) * 16);
#pragma unroll
                    for (int u = 0; u < NL; ++u)
                        if (v + 32 * u < v1)
                            count8(w[u]);
                }
                tail0 = v1 * 8;
            }
            for (int i = tail0 + lane; i < e1; i += 32)
                count(__ldg(reinterpret_cast<const unsigned short *>(slice.p) + i));
        }
        __syncthreads();
        // block totals, pushed into every block's gather slot of this rank: one cluster barrier
        for (int o = threadIdx.x; o < kFKeys; o += blockDim.x) {
            unsigned tot = 0;
            for (int ci = 0; ci < nck; ++ci)
                tot += U.k.hc[ci][o];
            for (int q = 0; q < csize; ++q)
                cluster.map_shared_rank(&U.k.gather[0][0], q)[rank * kFKeys + o] = tot;
            U.k.km[o] = (uint32_t)o < kmax ? fx(x_of<1>(kmax - (uint32_t)o)) : 0ull;
        }
        cluster.sync();
        for (int o = threadIdx.x; o < kFKeys; o += blockDim.x) {
            unsigned tot = 0;
            for (int q = 0; q < csize; ++q)
                tot += U.k.gather[q][o];
            U.k.bh[o] = tot;
        }
        __syncthreads();
#ifdef SPEC_FILTER_BLOCK_SELECT
        {
            bool ok = true;
            int pcut = kFKeys - 1;
            if (use_k) {
                find_crossing(S, kFKeys, 0ull, (unsigned long long)tk,
                              [&](int o) { return (unsigned long long)U.k.bh[o]; });
                ok = S.pos >= 0;
                pcut = S.pos;
            }
            if (ok && use_p) {
                unsigned long long target;
                const int pk = pcut;
                if (use_k) {
                    unsigned long long sk = 0;
                    for (int o = threadIdx.x; o <= pk; o += blockDim.x)
                        sk += (unsigned long long)U.k.bh[o] * U.k.km[o];
                    target = (unsigned long long)ceil((double)tp * (double)block_sum_u64(S, sk));
                } else {
                    target = (unsigned long long)ceil((double)tp * S.z);
                }
                find_crossing(S, kFKeys, 0ull, target,
                              [&](int o) { return o <= pk ? (unsigned long long)U.k.bh[o] * U.k.km[o] : 0ull; });
                if (S.pos >= 0)
                    pcut = S.pos;
                else
                    ok = use_k;
            }
            __syncthreads();
            if (threadIdx.x == 0)
                S.pos = ok ? pcut : -1;
        }
#else
        // selection by warp 0 alone (lanes own 16 consecutive offsets), published by one barrier
        if (warp == 0) {
            constexpr int PER = kFKeys / 32;
            // first offset o at which w(0) + ... + w(o) >= target (-1 if never), over o <= olim
            auto crossing = [&](unsigned long long target, int olim, bool by_mass) -> int {
                const int b0 = lane * PER;
                unsigned long long mine = 0;
#pragma unroll 4
                for (int k = 0; k < PER; ++k)
                    if (b0 + k <= olim)
                        mine += by_mass ? (unsigned long long)U.k.bh[b0 + k] * U.k.km[b0 + k]
                                        : (unsigned long long)U.k.bh[b0 + k];
                unsigned long long inc = mine;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long y = __shfl_up_sync(kFull, inc, o);
                    if (lane >= o)
                        inc += y;
                }
                unsigned long long c = inc - mine;
                int pos = -1;
                if (c < target && inc >= target)
                    for (int k = 0; k < PER; ++k) {
                        c += by_mass ? (unsigned long long)U.k.bh[b0 + k] * U.k.km[b0 + k]
                                     : (unsigned long long)U.k.bh[b0 + k];
                        if (c >= target) {
                            pos = b0 + k;
                            break;
                        }
                    }
                const unsigned found = __ballot_sync(kFull, pos >= 0);
                return found ? __shfl_sync(kFull, pos, __ffs(found) - 1) : -1;
            };
            bool ok = true;
            int pcut = kFKeys - 1;
            if (use_k) {
                pcut = crossing((unsigned long long)tk, kFKeys - 1, false);
                ok = pcut >= 0;  // fewer than k tokens in the window: the general path
            }
            if (ok && use_p) {
                unsigned long long target;
                if (use_k) {
                    unsigned long long sk = 0;
                    for (int o = lane; o <= pcut; o += 32)
                        sk += (unsigned long long)U.k.bh[o] * U.k.km[o];
                    target = (unsigned long long)ceil((double)tp * (double)warp_sum_u64(sk));
                } else {
                    target = (unsigned long long)ceil((double)tp * S.z);
                }
                const int pp2 = crossing(target, pcut, true);
                if (pp2 >= 0)
                    pcut = pp2;
                else
                    ok = use_k;  // with top-k every survivor is counted; top-p alone: the cut lies deeper
            }
            if (lane == 0)
                S.pos = ok ? pcut : -1;
        }
#endif
        __syncthreads();
        const int pcut = S.pos;
        if (pcut >= 0) {
            thr = kmax - (uint32_t)pcut;
            for (int ci = warp; ci < nck; ci += kFilterWarps) {
                const int c = c0 + ci;
                const float mk = S.cmax[ci];
                float mc = -INFINITY, sc = 0.f;
                if (mk > -INFINITY && key_of<1>(mk) >= thr) {
                    // s_c relative to the chunk maximum, from the row-relative fixed-point masses
                    mc = mk;
                    unsigned long long sum = 0;
                    for (int o = (int)(kmax - key_of<1>(mk)) + lane; o <= pcut; o += 32)
                        sum += (unsigned long long)U.k.hc[ci][o] * U.k.km[o];
                    sc = __ull2float_rn(warp_sum_u64(sum)) * kTwoM32 * ex2(M - mc * cs);
                }
                if (lane == 0)
                    pp[c] = make_float2(mc, sc);
            }
            done = true;
        }
        __syncthreads();  // the key counts are dead from here on
    }

    if (!done) {
        if (DT == 1)
            cluster.sync();  // every block is done with the one-pass arrays (the same storage)
        unsigned *cnt = U.g.cnt;
        auto binof = [&](float x) -> unsigned {  // round(d * kFBinScale), monotone; NaN and -inf last
            const float f = fmaf(-fmaf(x, cs, -M), kFBinScale, 12582912.f);
            return min(__float_as_uint(f) - 0x4B400000u, (unsigned)(kFBins - 1));
        };
        // least mass of a token of bin b (d <= (b + 1/2) / kFBinScale), with room for rounding
        auto lo_mass = [&](int b) -> unsigned long long {
            return b >= kFBins - 1 ? 0ull
                                   : __float2ull_rz(exp2f(-((float)b + 0.5f) / kFBinScale) * (4294967296.0f * 0.99998f));
        };

        // ---- 1. token counts per bin
        for (int b = threadIdx.x; b < kFBins; b += blockDim.x)
            cnt[b] = 0;
        __syncthreads();
        slice_for_each<DT>(slice, n, [&](float x, int) { atomicAdd(&cnt[binof(x)], 1u); });
        cluster_sum_hist(cnt, cluster, csize, kFBins);

        // ---- 2. the last bin that can hold a survivor
        int bk = kFBins;                // bin of the k-th largest logit (kFBins: no top-k)
        unsigned long long cabove = 0;  // tokens in the bins before bk
        int bhi;
        if (use_k) {
            find_crossing(S, kFBins, 0ull, (unsigned long long)tk, [&](int i) { return (unsigned long long)cnt[i]; });
            bk = S.pos < 0 ? kFBins - 1 : S.pos;
            cabove = S.pos < 0 ? 0ull : S.above;
            bhi = bk;
        } else {
            const unsigned long long target = (unsigned long long)ceil((double)tp * S.z);
            find_crossing(S, kFBins, 0ull, target, [&](int i) { return (unsigned long long)cnt[i] * lo_mass(i); });
            bhi = S.pos < 0 ? kFBins - 1 : S.pos;
        }
        unsigned long long nl = 0;
        for (int b = threadIdx.x; b <= bhi; b += blockDim.x)
            nl += cnt[b];
        const bool listed = block_sum_u64(S, nl) <= (unsigned long long)kFList;

        // scratch in U.g.local once the lists are merged (or when there are none)
        uint32_t *wkey = reinterpret_cast<uint32_t *>(U.g.local);       // window keys    [kFWindow]
        unsigned long long *wmass = U.g.local + kFWindow / 2;            // window weights [kFWindow]
        unsigned long long *dh = U.g.local + kFWindow / 2 + kFWindow;    // digit histogram [256]

        // The largest key K of the window with above + (weights of window keys >= K) >= target.
        auto rank_window = [&](unsigned long long above, unsigned long long target) {
            const int nw = min((int)S.nwin, kFWindow);
            if (threadIdx.x == 0)
                S.best = 0;
            __syncthreads();
            if ((int)threadIdx.x < nw) {
                const uint32_t ki = wkey[threadIdx.x];
                unsigned long long c = above;
                for (int j = 0; j < nw; ++j)
                    if (wkey[j] >= ki)
                        c += wmass[j];
                if (c >= target)
                    atomicMax(&S.best, ki);
            }
            __syncthreads();
            return S.best;
        };
        // The same over all the tokens of bin `bin` with key >= lo_key in the slice, by a radix
        // select on the order key (8-bit digits, one histogram pass each).
        auto select_in_bin = [&](int bin, uint32_t lo_key, unsigned long long above, unsigned long long target,
                                 bool by_mass) {
            uint32_t prefix = 0, pmask = 0;
            for (int shift = KEY_BITS - 8; shift >= 0; shift -= 8) {
                __syncthreads();
                for (int b = threadIdx.x; b < 256; b += blockDim.x)
                    dh[b] = 0;
                __syncthreads();
                slice_for_each<DT>(slice, n, [&](float x, int) {
                    const uint32_t key = key_of<DT>(x);
                    if (key >= lo_key && (key & pmask) == prefix && binof(x) == (unsigned)bin)
                        atomicAdd(&dh[(key >> shift) & 255u], by_mass ? fx(x) : 1ull);
                });
                cluster_sum_hist(dh, cluster, csize, 256);
                find_crossing(S, 256, above, target, [&](int i) { return dh[255 - i]; });
                const int pos = S.pos;
                if (pos >= 0)
                    above = S.above;
                prefix |= (pos < 0 ? 0u : 255u - (uint32_t)pos) << shift;
                pmask |= 255u << shift;
            }
            return prefix;
        };

        uint32_t tau = 0, lam = 0;
        if (listed) {
            // ---- 3. every token up to bin bhi into the cluster's candidate list
            if (threadIdx.x == 0)
                S.nlocal = 0;
            __syncthreads();
            slice_for_each<DT>(slice, n, [&](float x, int i) {
                if (binof(x) <= (unsigned)bhi) {
                    const unsigned j = atomicAdd(&S.nlocal, 1u);
                    if (j < (unsigned)kFList)
                        U.g.local[j] = ((unsigned long long)key_of<DT>(x) << 32) | (uint32_t)(lo + i);
                }
            });
            cluster.sync();  // every block's list is complete
            int off = 0;
            for (int q = 0; q < csize; ++q) {
                const int nq = min((int)*cluster.map_shared_rank(&S.nlocal, q), kFList - off);
                const unsigned long long *lq = cluster.map_shared_rank(U.g.local, q);
                for (int i = threadIdx.x; i < nq; i += blockDim.x)
                    U.g.list[off + i] = lq[i];
                off += nq;
            }
            if (threadIdx.x == 0)
                S.nlist = off;
            cluster.sync();  // every block has read every list: U.g.local is scratch from here on
            const int nlst = S.nlist;

            // gather the list's tokens of bin b with key >= lo_key into the window
            auto gather = [&](int b, uint32_t lo_key, bool by_mass) {
                if (threadIdx.x == 0)
                    S.nwin = 0;
                __syncthreads();
                for (int j = threadIdx.x; j < nlst; j += blockDim.x) {
                    const uint32_t key = (uint32_t)(U.g.list[j] >> 32);
                    const float x = x_of<DT>(key);
                    if (key >= lo_key && binof(x) == (unsigned)b) {
                        const unsigned w = atomicAdd(&S.nwin, 1u);
                        if (w < (unsigned)kFWindow) {
                            wkey[w] = key;
                            wmass[w] = by_mass ? fx(x) : 1ull;
                        }
                    }
                }
                __syncthreads();
            };

            // ---- 4. top-k
            if (use_k) {
                if (cnt[bk] <= (unsigned)kFWindow) {
                    gather(bk, 0u, false);
                    tau = rank_window(cabove, (unsigned long long)tk);
                } else {
                    tau = select_in_bin(bk, 0u, cabove, (unsigned long long)tk, false);
                }
            }
            // ---- 4. top-p
            if (use_p) {
                unsigned long long target;
                if (use_k) {
                    unsigned long long sk = 0;
                    for (int j = threadIdx.x; j < nlst; j += blockDim.x) {
                        const uint32_t key = (uint32_t)(U.g.list[j] >> 32);
                        if (key >= tau)
                            sk += fx(x_of<DT>(key));
                    }
                    target = (unsigned long long)ceil((double)tp * (double)block_sum_u64(S, sk));
                } else {
                    target = (unsigned long long)ceil((double)tp * S.z);
                }
                // exact bin masses of the listed survivors of top-k, as 16-bit halves
                unsigned *mlo = reinterpret_cast<unsigned *>(U.g.mh), *mhi = mlo + kFBins;
                __syncthreads();
                for (int b = threadIdx.x; b < 2 * kFBins; b += blockDim.x)
                    mlo[b] = 0;
                __syncthreads();
                for (int j = threadIdx.x; j < nlst; j += blockDim.x) {
                    const uint32_t key = (uint32_t)(U.g.list[j] >> 32);
                    if (key >= tau) {
                        const float x = x_of<DT>(key);
                        const unsigned long long w = fx(x);
                        const unsigned b = binof(x);
                        atomicAdd(&mlo[b], (unsigned)(w & 0xffffu));
                        atomicAdd(&mhi[b], (unsigned)(w >> 16));
                    }
                }
                __syncthreads();
                find_crossing(S, kFBins, 0ull, target,
                              [&](int i) { return ((unsigned long long)mhi[i] << 16) + (unsigned long long)mlo[i]; });
                const int bp = S.pos;
                const unsigned long long pabove = S.above;
                if (bp >= 0) {
                    if (cnt[bp] <= (unsigned)kFWindow) {
                        gather(bp, tau, true);
                        lam = rank_window(pabove, target);
                    } else {
                        lam = select_in_bin(bp, tau, pabove, target, true);
                    }
                }
            }
        } else {
            // ---- 3 / 4 over the slice: the list would be too long
            if (use_k)
                tau = select_in_bin(bk, 0u, cabove, (unsigned long long)tk, false);
            if (use_p) {
                unsigned long long target;
                if (use_k) {
                    unsigned long long sk = 0;
                    slice_for_each<DT>(slice, n, [&](float x, int) {
                        if (key_of<DT>(x) >= tau)
                            sk += fx(x);
                    });
                    target = (unsigned long long)ceil((double)tp * (double)cluster_sum_u64(S, cluster, csize, sk));
                } else {
                    target = (unsigned long long)ceil((double)tp * S.z);
                }
                __syncthreads();
                for (int b = threadIdx.x; b < kFBins; b += blockDim.x)
                    U.g.mh[b] = 0;
                __syncthreads();
                slice_for_each<DT>(slice, n, [&](float x, int) {
                    if (key_of<DT>(x) >= tau) {
                        const unsigned long long w = fx(x);
                        if (w)
                            atomicAdd(&U.g.mh[binof(x)], w);
                    }
                });
                cluster_sum_hist(U.g.mh, cluster, csize, kFBins);
                find_crossing(S, kFBins, 0ull, target, [&](int i) { return U.g.mh[i]; });
                const int bp = S.pos;
                const unsigned long long pabove = S.above;
                if (bp >= 0)
                    lam = select_in_bin(bp, tau, pabove, target, true);
            }
        }
        thr = max(max(tau, lam), 1u);

        // ---- 4. chunk partials over the survivors, in K1's format: the kept maximum of a chunk
        // is K1's chunk maximum when that survives (and the chunk has no survivor otherwise)
        for (int c = c0 + warp; c < c1; c += kFilterWarps) {
            const float mk = S.cmax[c - c0];
            float mc = -INFINITY, sc = 0.f;
            if (mk > -INFINITY && key_of<DT>(mk) >= thr) {
                mc = mk;
                const float Mc = mc * cs;
                unsigned long long sum = 0;
                if (listed) {
                    const uint32_t plo = (uint32_t)c * (uint32_t)P.chunk, phi = plo + (uint32_t)P.chunk;
                    for (int j = lane; j < S.nlist; j += 32) {
                        const unsigned long long e = U.g.list[j];
                        const uint32_t key = (uint32_t)(e >> 32), pos = (uint32_t)e;
                        if (pos >= plo && pos < phi && key >= thr)
                            sum += fx_chunk(x_of<DT>(key), Mc);
                    }
                } else {
                    const int64_t e0 = (int64_t)c * P.chunk - lo;
                    slice_range<DT>(slice, e0, min(n, e0 + P.chunk), lane, 32, [&](float x, int) {
                        if (key_of<DT>(x) >= thr)
                            sum += fx_chunk(x, Mc);
                    });
                }
                sc = __ull2float_rn(warp_sum_u64(sum)) * kTwoM32;
            }
            if (lane == 0)
                pp[c] = make_float2(mc, sc);
        }
    }
    if (rank == 0 && threadIdx.x == 0)
        P.thr[t] = thr;
    if (!done)
        cluster.sync();  // no block leaves while another may still read its shared memory (the
                         // one-pass path reads no other block's memory after its one barrier)
}

// ---------------------------------------------------------------------------------------
// Chunk combines (used by K2 / K4)
// ---------------------------------------------------------------------------------------

__device__ __forceinline__ int lane_combine_argmax(const Params &P, int64_t t, float *best_out)
{
    float best = -INFINITY;
    int idx = INT_MAX;
    const float2 *pp = P.part + t * P.nchunks;
    for (int c = 0; c < P.nchunks; ++c) {
        const float2 pc = pp[c];
        const int i = __float_as_int(pc.y);
        if (pc.x > best || (pc.x == best && i < idx)) {
            best = pc.x;
            idx = i;
        }
    }
    if (best_out)
        *best_out = best;
    return idx == INT_MAX ? 0 : idx;
}

// Warp combine of one row's softmax partials (lanes over chunks).
__device__ __forceinline__ void warp_combine_soft(const float2 *pp, int nchunks, float cs, int lane, float &M,
                                                  float &S)
{
    float m = -INFINITY;
    for (int c = lane; c < nchunks; c += 32) {
        const float x = pp[c].x;
        m = fmaxf(m, x);
    }
    m = warp_max(m);
    M = m * cs;
    float s = 0.f;
    if (m > -INFINITY) {
        for (int c = lane; c < nchunks; c += 32) {
            const float2 pc = pp[c];
            if (pc.x != -INFINITY)
                s += pc.y * ex2(pc.x * cs - M);
        }
    }
    S = warp_sum(s);
}

__device__ __forceinline__ int warp_combine_argmax(const float2 *pp, int nchunks, int lane)
{
    float best = -INFINITY;
    int idx = INT_MAX;
    for (int c = lane; c < nchunks; c += 32) {
        const float2 pc = pp[c];
        const int i = __float_as_int(pc.y);
        if (pc.x > best || (pc.x == best && i < idx)) {
            best = pc.x;
            idx = i;
        }
    }
    warp_argmax(best, idx);
    return idx == INT_MAX ? 0 : idx;
}

// ---------------------------------------------------------------------------------------
// K2: per-request finalize
// ---------------------------------------------------------------------------------------

template <int DT, bool F>
__global__ void __launch_bounds__(kThreads) finalize_kernel(Params P)
{
    allow_dependents();
    wait_for_prerequisite();  // the row statistics (and the cuts)
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (r >= P.B)
        return;
    const int errbits = P.err[0];
    if (errbits & SPEC_DEVERR_LAYOUT) {
        if (lane == 0) {
            P.out_acc[r] = -1;
            if (P.rstate) {
                P.rstate[r] = -1;
                P.rcnt[r] = 0;
            }
            if (P.dbg_z)
                P.dbg_z[r] = 0.f;
        }
        return;
    }
    const int cu0 = P.cu[r];
    const int k = P.cu[r + 1] - cu0;
    const int64_t tb = (int64_t)cu0 + r;
    const int64_t db = cu0;
    const bool too_long = k > SPEC_REJECT_MAX_SPEC_LEN;
    int xs = -1;
    if (!too_long && lane < k)
        xs = P.ids[db + lane];
    const unsigned badid = __ballot_sync(kFull, !too_long && lane < k && (xs < 0 || xs >= P.V));
    if (too_long || badid) {
        for (int64_t i = lane; i <= k; i += 32)
            P.out_tokens[tb + i] = -1;
        if (lane == 0) {
            P.out_acc[r] = -1;
            if (P.rstate) {
                P.rstate[r] = -1;
                P.rcnt[r] = 0;
            }
            if (P.dbg_z)
                P.dbg_z[r] = 0.f;
            atomicOr(P.err, too_long ? SPEC_DEVERR_SPEC_LEN : SPEC_DEVERR_DRAFT_ID);
            atomicMin(P.err + 1, r);
        }
        return;
    }

    const float temp = P.temp[r];
    const bool greedy = !(temp > 0.f);
    const float cs = greedy ? 0.f : kLog2e / temp;

    // Gathers of draft row `lane` that only need x*: issued before the partial combine.
    float ls = 0.f, qs = 1.f, ua = 0.f;
    uint32_t thr_i = 0;
    if (lane < k && !greedy) {
        if (P.thr)
            thr_i = P.thr[tb + lane];
        ls = load1<DT>(row_ptr<DT>(P, tb + lane), xs);
        if (P.q)
            qs = __ldg(P.q + (db + lane) * P.qstride + xs);
        ua = P.uni[2 * (tb + lane)];
    }

    // Row statistics of the draft rows, eight rows at a time: lanes run over the chunk
    // partials (coalesced, every load of the eight rows in flight together), then warp
    // reductions; lane i keeps row i's result.
    constexpr int G = 8;
    int am = 0;
    float Mi = -INFINITY, Si = 0.f;
    for (int i0 = 0; i0 < k; i0 += G) {
        float m[G], sv[G], best[G];
        int idx[G];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            m[j] = -INFINITY;
            sv[j] = 0.f;
            best[j] = -INFINITY;
            idx[j] = INT_MAX;
        }
        for (int c = lane; c < P.nchunks; c += 32) {
            float2 pc[G];
#pragma unroll
            for (int j = 0; j < G; ++j)
                pc[j] = (i0 + j < k) ? P.part[(tb + i0 + j) * P.nchunks + c] : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int j = 0; j < G; ++j) {
                if (greedy) {
                    const int ci = __float_as_int(pc[j].y);
                    if (pc[j].x > best[j] || (pc[j].x == best[j] && ci < idx[j])) {
                        best[j] = pc[j].x;
                        idx[j] = ci;
                    }
                } else if (pc[j].x != -INFINITY) {
                    const float Mc = pc[j].x * cs;
                    if (Mc > m[j]) {
                        sv[j] = (m[j] == -INFINITY) ? pc[j].y : sv[j] * ex2(m[j] - Mc) + pc[j].y;
                        m[j] = Mc;
                    } else {
                        sv[j] += pc[j].y * ex2(Mc - m[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < G; ++j) {
            if (greedy) {
                warp_argmax(best[j], idx[j]);
                if (lane == i0 + j)
                    am = idx[j] == INT_MAX ? 0 : idx[j];
            } else {
                const float mw = warp_max(m[j]);
                const float sw = warp_sum(m[j] == -INFINITY ? 0.f : sv[j] * ex2(m[j] - mw));
                if (lane == i0 + j) {
                    Mi = mw;
                    Si = sw;
                }
            }
        }
    }

    // Acceptance decision of draft row `lane`.
    bool accept = true;
    float wstar = 0.f;
    if (lane < k) {
        if (greedy) {
            accept = (xs == am);
        } else {
            const float e = fmaf(ls, cs, -Mi);  // x* is in Si unless the top-k / top-p cut removed it
            wstar = kept<DT, F>(ls, thr_i) ? ex2(e) : 0.f;
            const double lhs = (double)ua * (double)qs;  // exact
            const float ps = wstar / Si;
            if (ps > 1e-30f || wstar == 0.f)
                accept = lhs < (double)ps;
            else  // below fp32's normal range: form p(x*) in double
                accept = lhs < exp2((double)e) / (double)Si;
            if (P.dbg_pdraft)
                P.dbg_pdraft[db + lane] = ps;
        }
    }
    const unsigned rej = __ballot_sync(kFull, lane < k && !accept);
    const int j = rej ? __ffs(rej) - 1 : k;
    const int64_t tj = tb + j;

    int token = -1;
    bool pending = false;
    float zdbg = 0.f;
    if (greedy) {
        token = (j < k) ? __shfl_sync(kFull, am, j) : warp_combine_argmax(P.part + tj * P.nchunks, P.nchunks, lane);
    } else {
        const float us = P.uni[2 * tj + 1];
        const char *row = row_ptr<DT>(P, tj);
        const uint32_t thr = P.thr ? P.thr[tj] : 0u;
        if (j == k) {  // bonus: draw from p
            float M, S;
            warp_combine_soft(P.part + tj * P.nchunks, P.nchunks, cs, lane, M, S);
            ChunkMassFromPartials cm{P.part + tj * P.nchunks, cs, M, -1, 0.f};
            const float Z = chunk_total(cm, P.nchunks, lane);
            float th;
            const int c = chunk_locate(cm, P.nchunks, us * Z, lane, th);
            TargetMass<DT, F> f{row, cs, M, -1, thr};
            token = (int)warp_find(f, (int64_t)c * P.chunk, min((int64_t)P.V, (int64_t)(c + 1) * P.chunk), th, lane);
            zdbg = 1.f;
        } else {
            const float Mj = __shfl_sync(kFull, Mi, j);
            const float Sj = __shfl_sync(kFull, Si, j);
            const int xj = __shfl_sync(kFull, xs, j);
            if (!P.q) {  // one-hot draft: residual = p without x*
                // the chunk holding x*, summed again without it (no cancellation)
                const int cx = xj / P.chunk;
                TargetMass<DT, F> fx{row, cs, Mj, xj, thr};
                const float mx = warp_range_mass(fx, (int64_t)cx * P.chunk,
                                                 min((int64_t)P.V, (int64_t)(cx + 1) * P.chunk), lane);
                ChunkMassFromPartials cm{P.part + tj * P.nchunks, cs, Mj, cx, mx};
                float Z = chunk_total(cm, P.nchunks, lane);
                int64_t excl = xj;
                if (!(Z > 0.f)) {  // empty residual: draw from p itself
                    cm.override_chunk = -1;
                    Z = chunk_total(cm, P.nchunks, lane);
                    excl = -1;
                } else {
                    zdbg = Z / Sj;
                }
                float th;
                const int c = chunk_locate(cm, P.nchunks, us * Z, lane, th);
                TargetMass<DT, F> f{row, cs, Mj, excl, thr};
                token = (int)warp_find(f, (int64_t)c * P.chunk, min((int64_t)P.V, (int64_t)(c + 1) * P.chunk), th,
                                       lane);
            } else {  // explicit q: K3 / K4 finish this request
                pending = true;
                if (lane == 0)
                    P.rstat[r] = make_float2(Mj, Sj);
            }
        }
    }
    if (lane == 0) {
        P.out_acc[r] = j;
        if (P.rstate) {
            P.rstate[r] = pending ? j : -1;
            P.rcnt[r] = 0;
        }
        if (P.dbg_z && !pending)
            P.dbg_z[r] = zdbg;
    }
    if (P.counters) {  // this request's share of the acceptance counters (integer sums: order-free)
        unsigned long long *C = P.counters;
        if (lane == 0) {
            if (k > 0)
                atomicAdd(C + SPEC_METRIC_NUM_DRAFTS, 1ull);
            atomicAdd(C + SPEC_METRIC_NUM_DRAFT_TOKENS, (unsigned long long)k);
            atomicAdd(C + SPEC_METRIC_NUM_ACCEPTED_TOKENS, (unsigned long long)j);
            atomicAdd(C + SPEC_METRIC_NUM_VERIFIES, 1ull);
        }
        if (lane < j)
            atomicAdd(C + SPEC_METRIC_ACCEPTED_PER_POS + lane, 1ull);
    }
    for (int i = lane; i <= k; i += 32) {
        if (i == j && pending)
            continue;
        P.out_tokens[tb + i] = (i < j) ? xs : (i == j ? token : -1);
    }
}

// ---------------------------------------------------------------------------------------
// K3: explicit-q recovery, one block per request that rejected a draft
// ---------------------------------------------------------------------------------------

// Warps own contiguous ranges of (request, chunk) units; each unit's residual mass goes to
// rpart.  The warp that completes a request's last chunk (a per-request counter, zeroed by
// K2 in this same call) draws the recovered token from the chunk masses: chunk scan and
// warp descent as in K2.  No warp waits for another.
template <int DT, bool F>
__global__ void __launch_bounds__(kThreads, 4) residual_kernel(Params P)
{
    wait_for_prerequisite();  // the decisions (and the staged draft rows)
    const int lane = threadIdx.x & 31;
    const int64_t nunits = (int64_t)P.B * P.nchunks;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t per = (nunits + nw - 1) / nw;
    const int64_t u0 = gw * per;
    const int64_t u1 = min(nunits, u0 + per);
    for (int64_t u = u0; u < u1; ++u) {
        const int r = (int)(u / P.nchunks);
        const int c = (int)(u - (int64_t)r * P.nchunks);
        const int j = P.rstate[r];
        if (j < 0)
            continue;
        const int cu0 = P.cu[r];
        const int64_t t = (int64_t)cu0 + r + j;
        const int64_t d = (int64_t)cu0 + j;
        const float2 st = P.rstat[r];
        const float cs = kLog2e / P.temp[r];
        const char *row = row_ptr<DT>(P, t);
        const uint32_t thr = P.thr ? P.thr[t] : 0u;
        const ResidualMass<DT, F> f{row, P.q + d * P.qstride, cs, st.x, 1.f / st.y, thr};
        const float z = warp_residual_chunk(f, (int64_t)c * P.chunk, min((int64_t)P.V, (int64_t)(c + 1) * P.chunk),
                                            lane);
        int last = 0;
        if (lane == 0) {
            P.rpart[(int64_t)r * P.nchunks + c] = z;
            __threadfence();  // the mass is visible before the count says so
            last = atomicAdd(P.rcnt + r, 1) == P.nchunks - 1;
        }
        if (!__shfl_sync(kFull, last, 0))
            continue;
        __threadfence();
        const float us = P.uni[2 * t + 1];
        const ChunkMassFromL2 cmz{P.rpart + (int64_t)r * P.nchunks};
        const float Z = chunk_total(cmz, P.nchunks, lane);
        int token;
        if (Z > 0.f) {
            float th;
            const int cc = chunk_locate(cmz, P.nchunks, us * Z, lane, th);
            token = (int)warp_find(f, (int64_t)cc * P.chunk, min((int64_t)P.V, (int64_t)(cc + 1) * P.chunk), th, lane);
        } else {  // empty residual: draw from p itself
            const ChunkMassFromPartials cm{P.part + t * P.nchunks, cs, st.x, -1, 0.f};
            const float Zp = chunk_total(cm, P.nchunks, lane);
            float th;
            const int cc = chunk_locate(cm, P.nchunks, us * Zp, lane, th);
            const TargetMass<DT, F> ft{row, cs, st.x, -1, thr};
            token = (int)warp_find(ft, (int64_t)cc * P.chunk, min((int64_t)P.V, (int64_t)(cc + 1) * P.chunk), th,
                                   lane);
        }
        if (lane == 0) {
            P.out_tokens[t] = token;
            if (P.dbg_z)
                P.dbg_z[r] = Z > 0.f ? Z : 0.f;
        }
    }
}

// ---------------------------------------------------------------------------------------
// KL: calls without top-k / top-p, target rows read only up to each request's first rejection
// ---------------------------------------------------------------------------------------
//
// The acceptance test at draft position i needs target row t_i alone, and the test stops at
// the first rejection, so no row after it can change the result.  KL walks each request's
// rows in order: a block takes the next request from a queue, streams row t_i through its
// warps' TMA rings into chunk partials in shared memory (K1's per-unit reduction), decides
// position i with K2's arithmetic, and stops at the first rejection (or, every draft
// accepted, after the bonus row).  The output token is drawn in the same block: K2's chunk
// scan and warp descent, and for explicit draft probabilities K3's residual chunk masses over
// the rejected row, by all warps.  A request costs j + 1 target rows (j = its output
// position) and, on an explicit-q rejection, one draft row, where K1 / K3 read all k + 1
// target rows.  Every value that decides a token comes from the same functions as in K1, K2
// and K3, so the results are the same bit for bit.  Blocks never wait for one another.

constexpr int kLMaxChunks = (SPEC_REJECT_MAX_VOCAB * 4 + kUnitBytes - 1) / kUnitBytes;
#ifndef SPEC_KL_WARPS
#define SPEC_KL_WARPS 8       // warps per block, each with its own ring
#endif
#ifndef SPEC_KL_STAGES
#define SPEC_KL_STAGES 1      // ring slots per warp (8 warps x 2 blocks: 16 units in flight per SM)
#endif
#ifndef SPEC_KL_MIN_REQUESTS
#define SPEC_KL_MIN_REQUESTS 64  // smaller batches with cuts or host rows: the full pass is faster
#endif
#ifndef SPEC_KL_RESIDUAL_UNROLL
#define SPEC_KL_RESIDUAL_UNROLL 8  // 16-byte load groups in flight per lane in the residual pass (fp32 rows)
#endif
#ifndef SPEC_KL_RESIDUAL_UNROLL_BF16
#define SPEC_KL_RESIDUAL_UNROLL_BF16 16  // the same for bf16 rows without cuts (8 -> 16 took 1-2% off
                                         // large batches; with cuts 16 measured 2-4% slower)
#endif
#ifndef SPEC_KL_HOST_RESIDUAL_UNROLL
#define SPEC_KL_HOST_RESIDUAL_UNROLL 2  // the same, draft rows read over the host link (groups loaded before the copies are stored)
#endif
#ifndef SPEC_KL_MIN_BLOCKS
#define SPEC_KL_MIN_BLOCKS 2  // blocks per SM
#endif
#ifndef SPEC_KL_CLUSTER_LOG2
#define SPEC_KL_CLUSTER_LOG2 -1  // -1: cluster size by the rule below; 0..3: always 1, 2, 4 or 8 blocks
#endif

constexpr int kLWarps = SPEC_KL_WARPS;
constexpr int kLStages = SPEC_KL_STAGES;
constexpr int kLThreads = kLWarps * 32;
constexpr size_t kLSmem = (size_t)kLWarps * kLStages * kUnitBytes;
// The draw's block_find gives each thread 32 bytes of logits of the located chunk.
static_assert(kLThreads * 32 >= kUnitBytes, "a block of KL must cover a whole chunk in block_find");

// ---- KL with top-k / top-p (bf16 rows): the cut of one row, by the whole block
//
// The same cut as K1F, from the row KL has just streamed (its unfiltered chunk partials are in
// shared memory; the row is read again through the warp's ring slot, mostly from L2):
//   1. counts of tokens by order-key offset below the row maximum's key over a window of the
//      largest keys, tried in three widths: kCutNarrow (one binade of bf16; with at most
//      kCutNarrowChunks chunks, counted per chunk, and its tokens listed for the draw), kCutMid,
//      then kFKeys.  The first two mark their tokens with packed compares and count only those
//      (visit_marked); the widest counts every token (one histogram per warp, a sink per lane
//      for the rest).  Warp 0 finds the k-th largest key, S_k and the top-p key from the totals
//      (integer sums of count x fixed-point mass, K1F's one-pass rules).  A width is skipped
//      while the block's latest cut lay deeper (rows of a batch tend to cut alike);
//   2. partials over the survivors: from the per-chunk counts of the narrow window, else one more
//      pass adding, per kept token, the fixed-point mass of its key offset (K1F's count x mass sum);
//   3. a cut below the widest window is found by a radix select on the 16-bit order key (two
//      passes of digit histograms per selection), with the partials of K1F's general path.
// Whichever step finds it, the cut key and the partials are K1F's, bit for bit.

#ifndef SPEC_CUT_PARTS
#define SPEC_CUT_PARTS 2
#endif
constexpr int kCutParts = SPEC_CUT_PARTS;                 // a pass moves each chunk in this many copies,
constexpr int kCutPartBytes = kUnitBytes / kCutParts;     // of this size, all in flight at once
static_assert(kCutParts >= 2 && kCutParts <= 8 && kUnitBytes % (16 * kCutParts) == 0, "copies of whole vectors");
static_assert(kLStages == 1, "the passes of a cut use the warp's one ring slot as kCutParts parts");

constexpr int kCutNarrow = 128;       // largest keys counted per chunk first (one binade of bf16)
constexpr int kCutNarrowChunks = 64;  // chunks (4096 tokens) a row may have for the per-chunk counts
constexpr int kCutMid = 256;          // then the largest keys counted with marks (two binades)
static_assert(kCutMid + 32 <= kFKeys + 32 && kCutMid % 32 == 0 && (kCutMid / 32 & (kCutMid / 32 - 1)) == 0,
              "the middle window fits the per-warp histograms and splits evenly over a warp");
constexpr int kCutList = kFKeys - kCutNarrow;  // per warp: window tokens listed by the narrow count
                                               // (after its counts and a sink per lane)
constexpr int kKeptMax = 256;         // kept tokens an output row may have for the draw from the list
static_assert(kKeptMax < kCutList, "a warp lists every kept token of a row that keeps at most kKeptMax");
// A listed token names its chunk among its warp's (c = warp + nw * n) by n in bits 28-31: rows of
// up to kCutListChunks chunks can be listed (the 128-key count lists only rows of at most
// kCutNarrowChunks chunks).
constexpr int kCutListChunks = 16 * kLWarps;
static_assert(kCutNarrowChunks <= kCutListChunks, "the narrow count's rows fit the list format");
static_assert(kUnitBytes / 2 <= 4096, "a listed token's element in its chunk fits 12 bits");

struct CutSmem {
    unsigned hw[kLWarps][kFKeys + 32];                // per warp: tokens per key offset, then a sink per lane
    unsigned char hcc[kCutNarrowChunks][kCutNarrow];  // per chunk: tokens of the kCutNarrow largest keys
                                                      // (8 bits; hcc_over when a count did not fit)
    int hcc_over;
    unsigned bh[kFKeys];                // block totals per key offset
    unsigned long long km[kFKeys];      // fixed-point mass of one token per key offset
    union {
        unsigned long long bm[kFKeys];  // block masses per key offset (tokens x km)
        struct {                        // the draw from the list: kept tokens, in list order and sorted
            int idx[kKeptMax];
            float w[kKeptMax];
            int sidx[kKeptMax];
            float sw[kKeptMax];
        } kp;
    };
    unsigned long long rm[256];         // radix: weights per digit
    float cmx[kLMaxChunks];             // unfiltered chunk maxima
    unsigned long long red[kLWarps];
    double z;                           // normaliser (top-p alone), 2^-32 units
    float m;                            // row maximum
    int pos;                            // exact path: crossing offset (-1: fall back)
    int dsel;                           // radix: crossing digit (-1: none)
    unsigned long long dabove;
    int32_t tk;                         // the current request's top-k and top-p
    float tp;
    uint32_t thr;                       // cut key of the latest row (0 = none)
    int abort;                          // a copy of a pass did not land in time
    int ln[kLWarps];                    // per warp: window tokens its narrow count met (listed up to kCutList)
    int lok;                            // the latest cut's kept tokens are all listed (and at most kKeptMax)
    unsigned nkept;                     // the latest cut's kept tokens (from the window totals)
    int kc[kLWarps];                    // the draw from the list: kept tokens per warp
    int zok;                            // and whether its residual has mass
    int ktail;                          // and its kept tokens among the row's last V mod 8
    int tok;                            // and its token
    int narrow_miss;                    // the block's latest cut lay below the narrow window
    int mid_miss;                       // and below the middle one
    uint64_t bar[kLWarps][kCutParts];   // per warp: one mbarrier per part of its ring slot
    uint32_t ph[kLWarps];               // per warp: the parity each of them is waiting for (a bit each)
};
constexpr size_t kLCutSmem = kLSmem + sizeof(CutSmem);

// First position (in order 0, 1, ...) of 256 digit weights w at which above0 + cum >= target,
// by warp 0 (8 per lane); -1 if the total falls short.  Returns the position and the weight
// before it through C.dsel / C.dabove.
template <class WF>
__device__ __forceinline__ void warp_digit_crossing(CutSmem &C, unsigned long long above0, unsigned long long target,
                                                    WF w)
{
    const int lane = threadIdx.x & 31;
    const int b0 = lane * 8;
    unsigned long long mine = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        mine += w(b0 + k);
    unsigned long long inc = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(kFull, inc, o);
        if (lane >= o)
            inc += y;
    }
    unsigned long long c = above0 + inc - mine;
    int pos = -1;
    unsigned long long ab = 0;
    if (c < target && c + mine >= target)
        for (int k = 0; k < 8; ++k) {
            const unsigned long long wk = w(b0 + k);
            if (c + wk >= target) {
                pos = b0 + k;
                ab = c;
                break;
            }
            c += wk;
        }
    const unsigned found = __ballot_sync(kFull, pos >= 0);
    if (lane == 0)
        C.dsel = -1;
    __syncwarp();
    if (found && lane == __ffs(found) - 1) {
        C.dsel = pos;
        C.dabove = ab;
    }
}

// The bf16 pair holding twice the logit whose order key is `key` (keys under that of -inf,
// 0x80, are NaNs: a lower key gives -inf).
__device__ __forceinline__ uint32_t bf16_pair_of_key(uint32_t key)
{
    const uint32_t b = __float_as_uint(x_of<1>(key > 0x80u ? key : 0x80u)) >> 16;
    return b | (b << 16);
}

// The tokens of one copy in shared memory (nv 16-byte vectors of bf16; lane l takes vectors l,
// l + 32, ...) whose logits compare >= the pair lo2 (the order keys follow the logits: -0 and +0
// share a key and compare equal; NaN compares false).  A packed compare tests two tokens; the
// results of four vectors become a 32-bit mask per lane, and visit(bits, element, ballot) runs
// once per marked token, one per lane and turn, all lanes in step, so that the warp takes as many
// turns as its busiest lane has marks; turn(ballot) follows every turn.  Cheap where the marked
// tokens are few, as above a cut or inside a narrow window.
template <class Visit, class Turn>
__device__ __forceinline__ void visit_marked(const uint4 *st, int nv, uint32_t lo2, Visit visit, Turn turn)
{
    const int lane = threadIdx.x & 31;
    auto ge = [&](uint32_t x) {  // 0xffff per 16-bit half holding a logit >= lo2's
        uint32_t r;
        asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(lo2));
        return r;
    };
    auto mask8 = [&](const uint4 &x) -> uint32_t {  // bit e: element e of the vector is marked
        const uint32_t f0 = __byte_perm(ge(x.x), ge(x.y), 0x6420) & 0x01010101u;  // elements 0..3, a byte each
        const uint32_t f1 = __byte_perm(ge(x.z), ge(x.w), 0x6420) & 0x01010101u;  // elements 4..7
        return ((f0 * 0x01020408u) >> 24) | (((f1 * 0x01020408u) >> 20) & 0xf0u);  // bytes to bits
    };
    const unsigned short *st16 = reinterpret_cast<const unsigned short *>(st);
    for (int g = 0; g * 4 * 32 < nv; ++g) {  // uniform over the warp
        const int v0 = g * 4 * 32 + lane;
        uint32_t m = 0;
#pragma unroll
        for (int t = 0; t < 4; ++t)
            if (v0 + 32 * t < nv)
                m |= mask8(st[v0 + 32 * t]) << (8 * t);
        for (;;) {
            const unsigned bal = __ballot_sync(kFull, m != 0u);
            if (!bal)
                break;
            if (m) {
                const int b = __ffs(m) - 1;
                m &= m - 1;
                const int e = (v0 + 32 * (b >> 3)) * 8 + (b & 7);  // element of the copy
                visit((uint32_t)st16[e], e, bal);
            }
            turn(bal);
        }
    }
}

// Cut of row `row` of V logits in chunks of `chunk` at scale cs, with the request's top-k and
// top-p in C (all threads of the block; spart holds the row's unfiltered partials on entry and
// the partials over the survivors on return).  Leaves the cut key in C.thr (0: no cut).  The
// request's values stay in shared memory and the dimensions come by value, which keeps the
// caller's registers free for its streaming loop.
struct CutDims {
    int V, chunk, nchunks;
    int32_t *err;          // error word (a copy that does not land in time)
    unsigned char *slot;   // the warp's ring slot (free while the row is cut)
};
template <int DT>
__device__ __noinline__ uint32_t kl_cut_key(const CutDims P, CutSmem &C, float2 *spart, const char *row, float cs,
                                            int32_t tk, float tp, bool use_k)
{
    const bool use_p = tp > 0.f && tp < 1.f;
    constexpr int kB = kFKeys;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = (int)(blockDim.x >> 5);
    constexpr float kTwo32 = 4294967296.0f, kTwoM32f = 2.3283064365386963e-10f;

    // ---- row maximum and (top-p alone) the normaliser from the unfiltered partials (K1F)
    if (warp == 0) {
        float mm = -INFINITY;
        for (int c = lane; c < P.nchunks; c += 32)
            mm = fmaxf(mm, spart[c].x);
        mm = warp_max(mm);
        double z = 0.0;
        if (!use_k && mm > -INFINITY) {
            const float Mm = mm * cs;
            for (int c = lane; c < P.nchunks; c += 32) {
                const float2 pc = spart[c];
                if (pc.x != -INFINITY)
                    z += (double)pc.y * (double)ex2(pc.x * cs - Mm);
            }
            z = warp_sum_f64(z);
        }
        if (lane == 0) {
            C.m = mm;
            C.z = z * 4294967296.0;
        }
    }
    for (int c = threadIdx.x; c < P.nchunks; c += blockDim.x)
        C.cmx[c] = spart[c].x;
    for (int i = threadIdx.x; i < nw * (kB + 32); i += blockDim.x)
        (&C.hw[0][0])[i] = 0u;
    if (threadIdx.x == 0)
        C.hcc_over = 0;
    __syncthreads();
    const float m = C.m;
    if (!(m > -INFINITY))
        return 0u;  // no finite logit (the same for every thread): no cut
    const float M = m * cs;
    auto fx = [&](float x) -> unsigned long long { return __float2ull_rn(ex2(fmaf(x, cs, -M)) * kTwo32); };
    const uint32_t kmax = key_of<1>(m);
    const bool plain = kmax >= 0x8000u + (uint32_t)kB;
    auto offset = [&](uint32_t b16) -> uint32_t {  // key offset below kmax of the bf16 bits b16
        if (plain)
            return kmax - 0x8000u - b16;
        const uint32_t sg = (uint32_t)((int32_t)(b16 << 16) >> 31);
        return kmax - (0x8000u + (((b16 & 0x7fffu) ^ sg) - sg));
    };
    // A pass over this warp's chunks c = warp, warp + nw, ...: each chunk in kCutParts copies of
    // at most kCutPartBytes (TMA, into the parts of the warp's ring slot, all in flight), then
    // start(c), fv(st, nv, c, lo) for the nv 16-byte vectors st[] of each copy in shared memory,
    // elements lo, lo + 1, ... of the row (the warp's lanes take vectors lane, lane + 32, ...:
    // per_vec) and fe(bits)
    // for the last elements of the row past a multiple of 8 (global memory), then done(c).  Chunks with want(c) false are not
    // read (empty copies keep the barriers' phases in step).  A copy that does not land in time
    // sets C.abort; the pass still returns through every barrier of the block.
    auto pass = [&](auto want, auto start, auto fv, auto fe, auto done) {
        constexpr int kPart = kCutPartBytes / 2;  // bf16 elements per copy
        const int nmine = warp < P.nchunks ? (P.nchunks - 1 - warp) / nw + 1 : 0;
        const int n = kCutParts * nmine;
        uint32_t ph = C.ph[warp];
        auto range = [&](int u, int &c, int &lo, int &hi) {
            c = warp + nw * (u / kCutParts);
            const int c0 = c * P.chunk, c1 = min(P.V, c0 + P.chunk);
            lo = min(c1, c0 + (u % kCutParts) * kPart);
            hi = min(c1, lo + kPart);
        };
        auto issue = [&](int u) {  // lane 0
            int c, lo, hi;
            range(u, c, lo, hi);
            const uint32_t bytes = want(c) ? ((uint32_t)(hi - lo) * 2u) & ~15u : 0u;
            uint64_t *bar = &C.bar[warp][u % kCutParts];
            mbar_arrive_expect_tx(bar, bytes);
            if (bytes)
                bulk_g2s(P.slot + (u % kCutParts) * kCutPartBytes, row + (size_t)lo * 2, bytes, bar);
        };
        if (lane == 0)
            for (int u = 0; u < kCutParts && u < n; ++u)
                issue(u);
        for (int u = 0; u < n; ++u) {
            const int sl = u % kCutParts;
            if (!__all_sync(kFull, mbar_wait(&C.bar[warp][sl], (ph >> sl) & 1u, P.err))) {
                if (lane == 0) {  // let the copies still in flight land before the slot is reused
                    for (int u2 = u; u2 < u + kCutParts && u2 < n; ++u2)
                        mbar_wait(&C.bar[warp][u2 % kCutParts], (ph >> (u2 % kCutParts)) & 1u, P.err);
                    C.abort = 1;
                }
                break;
            }
            ph ^= 1u << sl;
            int c, lo, hi;
            range(u, c, lo, hi);
            if (want(c)) {
                if (sl == 0)
                    start(c);
                const uint4 *st = reinterpret_cast<const uint4 *>(P.slot + sl * kCutPartBytes);
                const int nv = (hi - lo) >> 3;
                fv(st, nv, c, lo);
                for (int i = lo + nv * 8 + lane; i < hi; i += 32)
                    fe((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(row) + i));
                if (sl == kCutParts - 1)
                    done(c);
            }
            __syncwarp();  // the part is consumed: refill it
            if (lane == 0 && u + kCutParts < n)
                issue(u + kCutParts);
        }
        if (lane == 0)
            C.ph[warp] = ph;
    };
    auto all = [](int) { return true; };
    auto nop = [](int) {};
    auto per_vec = [&](auto f) {
        return [&, f](const uint4 *st, int nv, int, int) {
            for (int v = lane; v < nv; v += 32)
                f(st[v]);
        };
    };
    auto each8 = [](const uint4 &w, auto fe) {
        fe(w.x & 0xffffu);
        fe(w.x >> 16);
        fe(w.y & 0xffffu);
        fe(w.y >> 16);
        fe(w.z & 0xffffu);
        fe(w.z >> 16);
        fe(w.w & 0xffffu);
        fe(w.w >> 16);
    };

    // block totals, one token's mass and the block masses for the offsets below n (all threads)
    auto totals = [&](int n, auto count) {
        for (int o = threadIdx.x; o < n; o += blockDim.x) {
            const unsigned tot = count(o);
            const unsigned long long km = (uint32_t)o < kmax ? fx(x_of<1>(kmax - (uint32_t)o)) : 0ull;
            C.bh[o] = tot;
            C.km[o] = km;
            C.bm[o] = (unsigned long long)tot * km;
        }
        __syncthreads();
    };
    auto select_window = [&](int win) {
    // ---- 2. selection by warp 0 over a window of n keys (lanes own n / 32 consecutive offsets),
    // K1F's one-pass rules; C.pos = the cut offset, or -1 when the cut lies below the window
    if (warp == 0) {
        const int n = win;
        const int PER = n / 32;  // a power of two
        // first offset o <= olim at which w(0) + ... + w(o) >= target (-1 if never)
        auto crossing = [&](unsigned long long target, int olim, bool by_mass) -> int {
            const int b0 = lane * PER;
            auto w = [&](int o) -> unsigned long long {
                return o > olim ? 0ull : by_mass ? C.bm[o] : (unsigned long long)C.bh[o];
            };
            unsigned long long mine = 0;
            for (int k = 0; k < PER; ++k)  // in a lane-rotated order: no shared-memory bank conflicts
                mine += w(b0 + ((k + lane) & (PER - 1)));
            unsigned long long inc = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(kFull, inc, o);
                if (lane >= o)
                    inc += y;
            }
            unsigned long long c = inc - mine;
            int pos = -1;
            if (c < target && inc >= target)
                for (int k = 0; k < PER; ++k) {
                    c += w(b0 + k);
                    if (c >= target) {
                        pos = b0 + k;
                        break;
                    }
                }
            const unsigned found = __ballot_sync(kFull, pos >= 0);
            return found ? __shfl_sync(kFull, pos, __ffs(found) - 1) : -1;
        };
        bool ok = true;
        int pcut = n - 1;
        if (use_k) {
            pcut = crossing((unsigned long long)tk, n - 1, false);
            ok = pcut >= 0;  // fewer than k tokens in the window
        }
        if (ok && use_p) {
            unsigned long long target;
            if (use_k) {
                unsigned long long sk = 0;
                for (int o = lane; o <= pcut; o += 32)
                    sk += C.bm[o];
                target = (unsigned long long)ceil((double)tp * (double)warp_sum_u64(sk));
            } else {
                target = (unsigned long long)ceil((double)tp * C.z);
            }
            const int p2 = crossing(target, pcut, true);
            if (p2 >= 0)
                pcut = p2;
            else
                ok = use_k;  // top-p alone: the cut lies below the window
        }
        if (lane == 0)
            C.pos = ok ? pcut : -1;
    }
    };

    // counts by key offset over the w largest keys in the warp's histogram: windows up to kCutMid
    // count their marked tokens only (visit_marked: about one token in a hundred for the narrow
    // window), wider ones every token, with a sink per lane for the tokens below the window (no
    // branch); with `flush`, the counts of each chunk move to C.hcc[c] after the chunk (8 bits
    // each; a larger count sets C.hcc_over) and the window's tokens are listed
    auto count_pass = [&](int w, bool flush) {
        unsigned *h = C.hw[warp];
        const uint32_t sink = (uint32_t)w + (uint32_t)lane;
        auto fe = [&](uint32_t b16) { atomicAdd(&h[min(offset(b16), sink)], 1u); };
        const bool marks = w <= kCutMid;
        const uint32_t lo2 = bf16_pair_of_key(kmax >= (uint32_t)(w - 1) ? kmax - (uint32_t)(w - 1) : 0u);
        // with `flush`, the window's tokens also go to the warp's list (while it has room): (the
        // warp's chunk number << 28) | (element in the chunk << 16) | bf16 bits
        uint32_t *list = C.hw[warp] + kCutNarrow + 32;
        int nl = 0;  // tokens met (every lane)
        const unsigned lt = (1u << lane) - 1u;
        auto vec = [&](const uint4 *st, int nv, int c, int lo) {
            if (!marks) {
                for (int v = lane; v < nv; v += 32)
                    each8(st[v], fe);
                return;
            }
            const uint32_t tag = ((uint32_t)((c - warp) / nw) << 28) | ((uint32_t)(lo - c * P.chunk) << 16);
            visit_marked(st, nv, lo2,
                         [&](uint32_t b16, int e, unsigned bal) {
                             atomicAdd(&h[offset(b16)], 1u);  // inside the window: below w
                             const int pos = nl + __popc(bal & lt);
                             if (flush && pos < kCutList)
                                 list[pos] = tag + ((uint32_t)e << 16) + b16;
                         },
                         [&](unsigned bal) { nl += __popc(bal); });
        };
        // a chunk whose maximum lies below the window holds no token of it: not read (its
        // per-chunk counts are zeros)
        auto reaches = [&](int c) {
            const float mk = C.cmx[c];
            return mk > -INFINITY && key_of<1>(mk) + (uint32_t)(w - 1) >= kmax;
        };
        if (flush)
            for (int c = warp; c < P.nchunks; c += nw)
                if (!reaches(c))
                    for (int o = lane; o < w; o += 32)
                        C.hcc[c][o] = 0;
        bool low = false;  // some chunk is skipped (else the pass takes every chunk without a test)
        for (int c = threadIdx.x; c < P.nchunks; c += blockDim.x)
            low = low || !reaches(c);
        low = __syncthreads_or(low);
        auto flush_chunk = [&](int c) {
            if (flush) {
                __syncwarp();  // every lane's counts of the chunk are in
                for (int o = lane; o < w; o += 32) {
                    const unsigned n = h[o];
                    C.hcc[c][o] = (unsigned char)min(n, 255u);
                    if (n > 255u)
                        C.hcc_over = 1;
                    h[o] = 0u;
                }
                __syncwarp();
            }
        };
        if (low)
            pass(reaches, nop, vec, fe, flush_chunk);
        else
            pass(all, nop, vec, fe, flush_chunk);
        if (flush && lane == 0)  // (the row's last elements past a multiple of 8 are counted, not listed)
            C.ln[warp] = nl;
        __syncthreads();
    };

    // ---- 1a. with at most kCutNarrowChunks chunks, first the kCutNarrow largest keys counted per
    // chunk: a cut inside them gets its partials from the counts, with no second pass.  (Skipped
    // while the block's latest cut lay deeper: rows of a batch tend to cut alike, and either
    // path gives the same key and partials.  A chunk with more than 255 tokens on one key of
    // the window takes the wide path too.)
    // Tokens the cut at offset p keeps (keys kmax - p .. kmax), from the latest window's totals.
    auto kept_count = [&](int p) -> unsigned {
        if (warp == 0) {
            unsigned t = 0;
            for (int o = lane; o <= p; o += 32)
                t += C.bh[o];
            t = __reduce_add_sync(kFull, t);
            if (lane == 0)
                C.nkept = t;
        }
        __syncthreads();
        return C.nkept;
    };
    // The output row's draw reads its kept tokens from a list (kl_list_draw) exactly when the cut
    // lies inside the widest window (any of the three finds it, by the block's history), keeps at
    // most kKeptMax tokens and the row has at most kCutListChunks chunks: a property of the row, so
    // the draw's arithmetic does not depend on which window the block tried.
    int pcut = -1;
    if (P.nchunks <= kCutNarrowChunks && !C.narrow_miss) {
        count_pass(kCutNarrow, true);
        int pn = -1;
        if (!C.hcc_over) {  // uniform: read after the pass's last barrier
            totals(kCutNarrow, [&](int o) {
                unsigned t = 0;
                for (int c = 0; c < P.nchunks; ++c)
                    t += C.hcc[c][o];
                return t;
            });
            select_window(kCutNarrow);
            __syncthreads();
            pn = C.pos;
        }
        bool narrow_done = false;
        if (pn >= 0) {
            const bool few = kept_count(pn) <= (unsigned)kKeptMax;
            bool listed = true;  // every warp's window tokens are in its list
            for (int w = 0; w < nw; ++w)
                listed = listed && C.ln[w] <= kCutList;
            if (few && !listed)
                pcut = pn;  // the listing pass below (the partials it gives are these, bit for bit)
            else
                narrow_done = true;
            if (threadIdx.x == 0)
                C.lok = few && listed;  // read after the barrier below
        }
        if (narrow_done) {  // K1F's one-pass partials
            const uint32_t thr = kmax - (uint32_t)pn;
            for (int c = warp; c < P.nchunks; c += nw) {
                const float mk = C.cmx[c];
                float mc = -INFINITY, sc = 0.f;
                if (mk > -INFINITY && key_of<1>(mk) >= thr) {
                    mc = mk;
                    unsigned long long sum = 0;
                    for (int o = lane; o <= pn; o += 32)
                        sum += (unsigned long long)C.hcc[c][o] * C.km[o];
                    sc = __ull2float_rn(warp_sum_u64(sum)) * kTwoM32f * ex2(M - mc * cs);
                }
                if (lane == 0)
                    spart[c] = make_float2(mc, sc);
            }
            __syncthreads();
            return thr;
        }
        if (pcut < 0) {
            for (int i = threadIdx.x; i < nw * (kB + 32); i += blockDim.x)
                (&C.hw[0][0])[i] = 0u;  // sinks of the narrow window sit inside the wide one
            if (threadIdx.x == 0)
                C.narrow_miss = 1;
            __syncthreads();
        }
    }

    // ---- 1b. counts over the kCutMid largest keys, with marks (skipped while the block's latest
    // cut lay deeper), then 1c. over the kFKeys largest keys, every token counted
    if (pcut < 0 && !C.mid_miss) {
        count_pass(kCutMid, false);
        totals(kCutMid, [&](int o) {
            unsigned t = 0;
            for (int w = 0; w < nw; ++w)
                t += C.hw[w][o];
            return t;
        });
        select_window(kCutMid);
        __syncthreads();
        pcut = C.pos;
        if (pcut < 0) {
            for (int i = threadIdx.x; i < nw * (kB + 32); i += blockDim.x)
                (&C.hw[0][0])[i] = 0u;  // sinks of the middle window sit inside the wide one
            if (threadIdx.x == 0)
                C.mid_miss = 1;
            __syncthreads();
        }
    }
    if (pcut < 0) {
        count_pass(kB, false);
        totals(kB, [&](int o) {
            unsigned t = 0;
            for (int w = 0; w < nw; ++w)
                t += C.hw[w][o];
            return t;
        });
        select_window(kB);
        __syncthreads();
        pcut = C.pos;
    }
    if (threadIdx.x == 0 && pcut >= 0) {  // a cut that would have fit a skipped window: try it again
        if (pcut < kCutNarrow)
            C.narrow_miss = 0;
        if (pcut < kCutMid)
            C.mid_miss = 0;
    }
    if (pcut >= 0) {
        // ---- 3. chunk partials over the survivors: per kept token (marked against the cut key)
        // the fixed-point mass of its key offset, summed as integers, rescaled to the chunk maximum;
        // with at most kKeptMax kept tokens the pass also lists them for the draw (a warp lists at
        // most that many, well inside its room)
        const uint32_t thr = kmax - (uint32_t)pcut;
        const uint32_t thr2 = bf16_pair_of_key(thr);
        const bool listing = kept_count(pcut) <= (unsigned)kKeptMax && P.nchunks <= kCutListChunks;
        auto live = [&](int c) { return C.cmx[c] > -INFINITY && key_of<1>(C.cmx[c]) >= thr; };
        for (int c = warp; c < P.nchunks; c += nw)
            if (lane == 0 && !live(c))
                spart[c] = make_float2(-INFINITY, 0.f);
        unsigned long long sum = 0;
        uint32_t *list = C.hw[warp] + kCutNarrow + 32;
        int nl = 0;
        const unsigned lt = (1u << lane) - 1u;
        uint32_t tag = 0;
        auto add = [&](uint32_t b16, int e, unsigned bal) {
            sum += C.km[offset(b16)];
            if (listing) {
                const int pos = nl + __popc(bal & lt);
                if (pos < kCutList)
                    list[pos] = tag + ((uint32_t)e << 16) + b16;
            }
        };
        auto turn = [&](unsigned bal) { nl += __popc(bal); };
        auto fe = [&](uint32_t b16) {
            if (offset(b16) <= (uint32_t)pcut)
                sum += C.km[offset(b16)];
        };
        pass(live, nop,
             [&](const uint4 *st, int nv, int c, int lo) {
                 tag = ((uint32_t)((c - warp) / nw) << 28) | ((uint32_t)(lo - c * P.chunk) << 16);
                 visit_marked(st, nv, thr2, add, turn);
             },
             fe, [&](int c) {
                 const float mc = C.cmx[c];
                 const float sc = __ull2float_rn(warp_sum_u64(sum)) * kTwoM32f * ex2(M - mc * cs);
                 if (lane == 0)
                     spart[c] = make_float2(mc, sc);
                 sum = 0;
             });
        if (lane == 0)
            C.ln[warp] = nl;
        if (threadIdx.x == 0)
            C.lok = listing;  // (nl <= kKeptMax < kCutList in every warp)
        __syncthreads();
        return thr;
    }

    // ---- cut below the window: radix selects on the order key (high byte, then low byte)
    auto key16 = [](uint32_t b16) -> uint32_t {
        const uint32_t sg = (uint32_t)((int32_t)(b16 << 16) >> 31);
        return 0x8000u + (((b16 & 0x7fffu) ^ sg) - sg);
    };
    // The largest key K >= lo with (weights of the keys in [K, ...) that are >= lo) >= target,
    // 0 when the total falls short.  Weights: 1 per token, or its fixed-point mass.  With
    // p_of_total the target is ceil(tp * total weight), the total taken from the first level.
    auto select = [&](uint32_t lo, unsigned long long target, bool by_mass, bool p_of_total) -> uint32_t {
        uint32_t prefix = 0;
        unsigned long long above = 0;
        for (int level = 0; level < 2; ++level) {
            const int shift = level ? 0 : 8;
            for (int i = threadIdx.x; i < nw * (kB + 32); i += blockDim.x)
                (&C.hw[0][0])[i] = 0u;
            __syncthreads();
            unsigned *hc = C.hw[warp];
            unsigned long long *hm = reinterpret_cast<unsigned long long *>(C.hw[warp]);
            auto fe = [&](uint32_t b16) {
                const uint32_t key = key16(b16);
                if (key >= lo && (level == 0 || (key >> 8) == (prefix >> 8))) {
                    const uint32_t d = (key >> shift) & 255u;
                    if (by_mass) {
                        const unsigned long long w = fx(__uint_as_float(b16 << 16));
                        if (w)
                            atomicAdd(&hm[d], w);
                    } else {
                        atomicAdd(&hc[d], 1u);
                    }
                }
            };
            pass(all, nop, per_vec([&](const uint4 &w) { each8(w, fe); }), fe, nop);
            __syncthreads();
            for (int d = threadIdx.x; d < 256; d += blockDim.x) {
                unsigned long long t = 0;
                for (int w = 0; w < nw; ++w)
                    t += by_mass ? reinterpret_cast<const unsigned long long *>(C.hw[w])[d]
                                 : (unsigned long long)C.hw[w][d];
                C.rm[d] = t;
            }
            __syncthreads();
            if (warp == 0) {
                if (level == 0 && p_of_total) {
                    unsigned long long t = 0;
                    for (int d = lane; d < 256; d += 32)
                        t += C.rm[d];
                    target = (unsigned long long)ceil((double)tp * (double)warp_sum_u64(t));
                }
                warp_digit_crossing(C, above, target, [&](int i) { return C.rm[255 - i]; });
            }
            __syncthreads();
            if (C.dsel < 0)
                return 0u;  // uniform over the block
            above = C.dabove;
            prefix |= (255u - (uint32_t)C.dsel) << shift;
            __syncthreads();  // C.dsel is rewritten by the next level
        }
        return prefix;
    };
    uint32_t tau = 0, lam = 0;
    if (use_k)
        tau = select(0u, (unsigned long long)tk, false, false);
    if (use_p) {
        const unsigned long long target = use_k ? 0ull : (unsigned long long)ceil((double)tp * C.z);
        lam = select(tau, target, true, use_k);
    }
    const uint32_t thr = max(max(tau, lam), 1u);

    // ---- chunk partials over the survivors, relative to each chunk's maximum (K1F's general path)
    auto live = [&](int c) { return C.cmx[c] > -INFINITY && key_of<1>(C.cmx[c]) >= thr; };
    for (int c = warp; c < P.nchunks; c += nw)
        if (lane == 0 && !live(c))
            spart[c] = make_float2(-INFINITY, 0.f);
    unsigned long long sum = 0;
    float Mc = 0.f;  // the chunk's maximum, scaled
    auto fe = [&](uint32_t b16) {
        if (key16(b16) >= thr)
            sum += __float2ull_rn(ex2(fmaf(__uint_as_float(b16 << 16), cs, -Mc)) * kTwo32);
    };
    pass(live, [&](int c) { Mc = C.cmx[c] * cs; }, per_vec([&](const uint4 &w) { each8(w, fe); }), fe,
         [&](int c) {
             const float sc = __ull2float_rn(warp_sum_u64(sum)) * kTwoM32f;
             if (lane == 0)
                 spart[c] = make_float2(C.cmx[c], sc);
             sum = 0;
         });
    __syncthreads();
    return thr;
}

template <int DT> __device__ __noinline__ void kl_cut_row(const CutDims P, CutSmem &C, float2 *spart, const char *row, float cs)
{
    const int32_t tk = C.tk;
    const float tp = C.tp;
    const bool use_k = tk > 0 && tk < P.V;
    const bool use_p = tp > 0.f && tp < 1.f;
    if (threadIdx.x == 0)
        C.lok = 0;  // set by a cut whose window tokens are all listed (every other thread reads it
                    // after the cut's barriers, or after the caller's when there is no cut)
    if (!(use_k || use_p))
        return;  // C.thr stays 0
    const uint32_t thr = kl_cut_key<DT>(P, C, spart, row, cs, tk, tp, use_k);
    if (threadIdx.x == 0)
        C.thr = thr;
    __syncthreads();
}

// The output token of a cut row from the window tokens its narrow count listed (C.lok): every
// token the cut keeps (key >= C.thr) is among them, and every other token has no mass, so the
// draw reads the kept tokens only (and q at those tokens only) instead of the whole row.  The
// draw is the full path's: the smallest token whose cumulative mass, in token order, exceeds
// u * Z; the last token with mass when rounding leaves u * Z at or past the total.  Masses:
//   mode 0 (explicit q):  max(0, p(x) - q(x)), p(x) = 2^(x cs - M) / S (inv_s = 1 / S);
//   mode 1 (one-hot draft): 2^(x cs - M), none at x* (p without the draft token);
//   mode 2 (the bonus row): 2^(x cs - M);
// an empty residual (modes 0 and 1) draws from 2^(x cs - M).  All threads of the block; returns
// the token, or -1 when more than kKeptMax tokens are kept (the caller takes the full path).
__device__ __noinline__ int kl_list_draw(CutSmem &C, int chunk, int mode, const float *qrow, float cs, float M,
                                         float inv_s, int xstar, float u, const char *row, int V)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = (int)(blockDim.x >> 5);
    const unsigned lt = (1u << lane) - 1u;
    const uint32_t thr = C.thr;
    const uint32_t *list = C.hw[warp] + kCutNarrow + 32;
    const int n = C.ln[warp];
    auto key = [](uint32_t b16) {
        const uint32_t sg = (uint32_t)((int32_t)(b16 << 16) >> 31);
        return 0x8000u + (((b16 & 0x7fffu) ^ sg) - sg);
    };
    int cnt = 0;
    for (int i = lane; i < n; i += 32)
        cnt += key(list[i] & 0xffffu) >= thr;
    cnt = __reduce_add_sync(kFull, cnt);
    if (lane == 0)
        C.kc[warp] = cnt;
    // the row's last V mod 8 tokens (past a multiple of 8) are counted by the passes, not listed
    const int ntail = V & 7;
    const int tail0 = V - ntail;
    uint32_t tb = 0;
    bool tkeep = false;
    if (warp == 0) {
        if (lane < ntail) {
            tb = (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(row) + tail0 + lane);
            tkeep = key(tb) >= thr;
        }
        const unsigned tbal = __ballot_sync(kFull, tkeep);
        if (lane == 0)
            C.ktail = __popc(tbal);
    }
    __syncthreads();
    int off = 0, total = C.ktail, listed_total = 0;
    for (int w = 0; w < nw; ++w) {
        off += w < warp ? C.kc[w] : 0;
        listed_total += C.kc[w];
    }
    total += listed_total;
    if (total > kKeptMax || total == 0)
        return -1;  // uniform
    // the kept tokens with 2^(x cs - M), in list order (warp by warp)
    for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const uint32_t e = i < n ? list[i] : 0u;
        const bool keep = i < n && key(e & 0xffffu) >= thr;
        const unsigned bal = __ballot_sync(kFull, keep);
        if (keep) {
            const int pos = off + __popc(bal & lt);
            C.kp.idx[pos] = (warp + nw * (int)(e >> 28)) * chunk + (int)((e >> 16) & 0xfffu);
            C.kp.w[pos] = ex2(fmaf(__uint_as_float((e & 0xffffu) << 16), cs, -M));
        }
        off += __popc(bal);
    }
    if (warp == 0) {  // the kept tail tokens after the listed ones
        const unsigned bal = __ballot_sync(kFull, tkeep);
        if (tkeep) {
            const int pos = listed_total + __popc(bal & lt);
            C.kp.idx[pos] = tail0 + lane;
            C.kp.w[pos] = ex2(fmaf(__uint_as_float(tb << 16), cs, -M));
        }
    }
    __syncthreads();
    // sorted by token (the kept tokens are distinct; rank = kept tokens before it), with their
    // masses, or with p's when `with_p`
    auto sort = [&](bool with_p) {
        for (int t = threadIdx.x; t < total; t += blockDim.x) {
            const int x = C.kp.idx[t];
            const float p = C.kp.w[t];
            int rank = 0;
            for (int o = 0; o < total; ++o)
                rank += C.kp.idx[o] < x;
            C.kp.sidx[rank] = x;
            C.kp.sw[rank] = (with_p || mode == 2) ? p
                            : mode == 0         ? fmaxf(0.f, p * inv_s - __ldg(qrow + x))
                                                : (x == xstar ? 0.f : p);
        }
        __syncthreads();
    };
    // warp 0: lane l takes sorted tokens [b0, b1); seg = their mass, inc = the inclusive scan of
    // the segments, Z = the total
    const int per = (total + 31) / 32;
    const int b0 = min(total, lane * per), b1 = min(total, b0 + per);
    auto scan = [&](float &seg, float &inc) {
        seg = 0.f;
        for (int t = b0; t < b1; ++t)
            seg += C.kp.sw[t];
        inc = seg;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(kFull, inc, o);
            if (lane >= o)
                inc += y;
        }
        return __shfl_sync(kFull, inc, 31);
    };
    sort(false);
    if (mode != 2) {
        if (warp == 0) {
            float seg, inc;
            const float Z = scan(seg, inc);
            if (lane == 0)
                C.zok = Z > 0.f;
        }
        __syncthreads();
        if (!C.zok)  // empty residual: draw from p (uniform)
            sort(true);
    }
    if (warp == 0) {
        float seg, inc;
        const float Z = scan(seg, inc);
        const float th = u * Z;
        float run = inc - seg;
        int hit = -1;
        for (int t = b0; t < b1; ++t) {
            run += C.kp.sw[t];
            if (run > th) {
                hit = t;
                break;
            }
        }
        const unsigned found = __ballot_sync(kFull, hit >= 0);
        int t;
        if (found) {
            t = __shfl_sync(kFull, hit, __ffs(found) - 1);
        } else {  // rounding left u * Z at or past the total: the last token with mass
            int last = -1;
            for (int q = b0; q < b1; ++q)
                if (C.kp.sw[q] > 0.f)
                    last = q;
            t = (int)__reduce_max_sync(kFull, (unsigned)(last + 1)) - 1;
        }
        if (lane == 0)
            C.tok = t >= 0 ? C.kp.sidx[t] : (total > 0 ? C.kp.sidx[total - 1] : 0);
    }
    __syncthreads();
    const int token = C.tok;
    __syncthreads();  // C.tok and the kept arrays are rewritten by the next draw
    return token;
}



// Layout check and request-queue reset before KL (one block).
__global__ void __launch_bounds__(256) lazy_init_kernel(Params P)
{
    allow_dependents();
    validate_layout(P);
    if (threadIdx.x == 0) {
        P.err[2] = 0;  // next request to hand out (first-rejection pass)
        P.err[3] = 0;  // the same for a second, chained launch of it
    }
}

struct ChunkMassFromShared {  // chunk masses already reduced into shared memory
    const float *z;
    __device__ __forceinline__ float operator()(int c) const { return z[c]; }
};

// Cluster helpers of the clustered first-rejection pass (CS blocks per request).  With CS = 1
// they reduce to the block's own shared memory and __syncthreads().
template <int CS> __device__ __forceinline__ void cluster_barrier()
{
    if constexpr (CS > 1)
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    else
        __syncthreads();
}

template <int CS> __device__ __forceinline__ unsigned cluster_rank()
{
    if constexpr (CS > 1) {
        unsigned r;
        asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
        return r;
    } else {
        return 0;
    }
}

// The same shared variable in block `rank` of the cluster (generic address).
template <int CS, class T> __device__ __forceinline__ T *in_block(T *p, unsigned rank)
{
    if constexpr (CS > 1)
        return cg::this_cluster().map_shared_rank(p, rank);
    else
        return p;
}

// HOST: the target rows live in pinned host memory (read over the host link with 16-byte loads,
// sixteen in flight per lane) instead of device memory (TMA bulk copies).  CUT (bf16 rows): the
// call has top-k / top-p cuts, applied to each row as it is reached (rows in host memory are cut
// from their device copies).
// CS > 1: a thread-block cluster of CS blocks works on each request.  Its CS * kLWarps warps
// split every row and every residual pass (chunk c goes to cluster warp c mod (CS * kLWarps)),
// write their chunk partials and residual masses into the leader block's (rank 0) shared
// memory, and the leader's warp 0 decides and draws; the leader claims the requests and
// sends the request index and each decision to every block of the cluster.  Every block
// takes the same cluster barriers in the same order.
template <int DT, bool HOST, bool CUT, int CS = 1>
__global__ void __launch_bounds__(kLThreads, SPEC_KL_MIN_BLOCKS) lazy_kernel(Params P)
{
    static_assert(!CUT || DT == 1, "cuts in KL: bf16 rows (from host memory: through their device copies)");
    static_assert(CS == 1 || (!HOST && !CUT), "clusters: rows in device memory, no cuts");
    constexpr int ES = Elem<DT>::kSize;
    extern __shared__ __align__(128) unsigned char ring[];
    CutSmem &C = *reinterpret_cast<CutSmem *>(ring + kLSmem);  // CUT only: after the rings
    __shared__ __align__(8) uint64_t full[kLWarps * kLStages];
    __shared__ float2 spart[kLMaxChunks];  // chunk partials of the row just streamed
    __shared__ float srm[kLMaxChunks];     // residual chunk masses (explicit q)
    __shared__ int s_r, s_go, s_abort;
    __shared__ float s_M, s_S;
    __shared__ BlockSearch bsearch;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned rank = cluster_rank<CS>();
    const bool leader = rank == 0;
    const int cw = (int)rank * kLWarps + warp;  // this warp's index in the cluster
    constexpr int kCW = CS * kLWarps;           // warps per cluster
    float2 *const lpart = in_block<CS>(spart, 0u);  // the leader's chunk partials
    float *const lrm = in_block<CS>(srm, 0u);       // and residual masses

    if (P.wait_prior)
        wait_for_prerequisite();
    allow_dependents();  // a chained launch may take SM slots as this launch's blocks finish
    if (P.err[0] & SPEC_DEVERR_LAYOUT) {  // the whole batch is invalid (as K2 reports it)
        for (int r = P.r_begin + (int)(blockIdx.x * blockDim.x + threadIdx.x); r < P.r_end;
             r += gridDim.x * blockDim.x)
            P.out_acc[r] = -1;
        if (!P.wait_prior)
            wait_for_prerequisite();  // end after the launch this one is chained to (see the end)
        return;
    }
    if (threadIdx.x < kLWarps * kLStages)
        mbar_init(&full[threadIdx.x], 1);
    if constexpr (CUT) {
        if (threadIdx.x < kCutParts * kLWarps)
            mbar_init(&C.bar[0][0] + threadIdx.x, 1);
        if (threadIdx.x < kLWarps)
            C.ph[threadIdx.x] = 0;
        if (threadIdx.x == 0) {
            C.abort = 0;
            C.narrow_miss = 0;
            C.mid_miss = 0;
        }
    }
    mbar_fence_init();
    if (threadIdx.x == 0)
        s_abort = 0;
    cluster_barrier<CS>();  // every block's shared state is set up before any block writes into it
    unsigned char *slots = ring + (size_t)warp * kLStages * kUnitBytes;
    uint64_t *bars = full + warp * kLStages;
    int64_t qi = 0, qc = 0;  // this warp's units issued (lane 0) and consumed; slot = count % stages

    auto issue = [&](const char *row, int c) {
        const int s = (int)(qi % kLStages);
        const int64_t lo = (int64_t)c * P.chunk;
        const int64_t hi = min((int64_t)P.V, lo + P.chunk);
        const uint32_t bytes = (uint32_t)((hi - lo) * ES) & ~15u;
        mbar_arrive_expect_tx(&bars[s], bytes);
        if (bytes)
            bulk_g2s(slots + (size_t)s * kUnitBytes, row + lo * ES, bytes, &bars[s]);
        ++qi;
    };

    for (;;) {
        if (leader && threadIdx.x == 0) {
            const int nr = s_abort ? P.r_end : P.r_begin + atomicAdd(P.err + P.qslot, 1);
            for (unsigned q = 0; q < (unsigned)CS; ++q)
                *in_block<CS>(&s_r, q) = nr;
        }
        cluster_barrier<CS>();
        const int r = s_r;
        if (r >= P.r_end || (CS == 1 && s_abort))
            break;  // uniform across the cluster
        const int cu0 = P.cu[r];
        const int k = P.cu[r + 1] - cu0;
        const int64_t tb = (int64_t)cu0 + r;
        const int64_t db = cu0;
        // per-request checks, as K2 (every warp reads the same ids, so every warp agrees)
        const bool too_long = k > SPEC_REJECT_MAX_SPEC_LEN;
        int xs = -1;
        if (!too_long && lane < k)
            xs = P.ids[db + lane];
        const unsigned badid = __ballot_sync(kFull, !too_long && lane < k && (xs < 0 || xs >= P.V));
        if (too_long || badid) {
            if (leader && warp == 0) {
                for (int64_t i = lane; i <= k; i += 32)
                    P.out_tokens[tb + i] = -1;
                if (lane == 0) {
                    P.out_acc[r] = -1;
                    atomicOr(P.err, too_long ? SPEC_DEVERR_SPEC_LEN : SPEC_DEVERR_DRAFT_ID);
                    atomicMin(P.err + 1, r);
                }
            }
            cluster_barrier<CS>();  // s_r is rewritten for the next request
            continue;
        }
        const float temp = P.temp[r];
        const bool greedy = !(temp > 0.f);
        const float cs = greedy ? 0.f : kLog2e / temp;
        if constexpr (CUT)
            if (threadIdx.x == 0) {  // read by the cut after the first row's barrier
                C.tk = P.top_k ? P.top_k[r] : 0;
                C.tp = P.top_p ? P.top_p[r] : 1.f;
                C.thr = 0;
            }
        // inputs of the acceptance test of draft position `lane` (warp 0), issued first
        float ls = 0.f, qs = 1.f, ua = 0.f;
        if (leader && warp == 0 && !greedy) {
            if (lane < k) {
                ls = load1<DT>(row_ptr<DT>(P, tb + lane), xs);
                if (P.q)
                    qs = __ldg(P.q + (db + lane) * P.qstride + xs);
                ua = P.uni[2 * (tb + lane)];
            }
        }

        int j = k;       // output position: the first rejection, else the bonus row
        int am = 0;      // argmax of the latest row (greedy)
        float Mi = 0.f, Si = 0.f;
        for (int i = 0; i <= k; ++i) {
            const char *row = row_ptr<DT>(P, tb + i);
            // ---- stream row t_i: this warp's units c = cw, cw + kCW, ...
            int ci = cw;
            if (!HOST && lane == 0)
                for (int s = 0; s < kLStages && ci < P.nchunks; ++s, ci += kCW)
                    issue(row, ci);
            bool ok = true;
            if constexpr (HOST) {
                for (int c = warp; c < P.nchunks; c += kLWarps) {
                    UnitRange R;
                    R.lo = (int64_t)c * P.chunk;
                    R.hi = min((int64_t)P.V, R.lo + P.chunk);
                    R.vlo = R.lo;
                    R.nvec = ((R.hi - R.lo) * ES) / 16;
                    R.vhi = R.vlo + R.nvec * Elem<DT>::kVec;
                    const char *u0 = row + R.lo * ES;
                    uint4 v[kVecPerLane];
#pragma unroll
                    for (int kk = 0; kk < kVecPerLane; ++kk) {
                        const int vi = kk * 32 + lane;
                        v[kk] = (vi < R.nvec) ? ld_stream(u0 + (size_t)vi * 16) : neg_inf_vec<DT>();
                    }
                    if (P.lstage) {  // the device copy of the row, for the residual pass and the draw
                        char *d0 = P.lstage + (size_t)(tb + i) * P.lstride * ES + R.lo * ES;
#pragma unroll
                        for (int kk = 0; kk < kVecPerLane; ++kk) {
                            const int vi = kk * 32 + lane;
                            if (vi < R.nvec)
                                *reinterpret_cast<uint4 *>(d0 + (size_t)vi * 16) = v[kk];
                        }
                        for (int64_t e = R.vhi + lane; e < R.hi; e += 32)
                            for (int b = 0; b < ES; ++b)
                                d0[(e - R.lo) * ES + b] = row[e * ES + b];
                    }
                    if (greedy)
                        argmax_regs<DT>(&spart[c], lane, v, R, row);
                    else
                        softmax_regs<DT>(&spart[c], cs, lane, v, R, row);
                }
                if (CUT && P.lstage)  // the cut reads the device copy through the bulk-copy engine
                    fence_proxy_async_global();
            } else
            for (int c = cw; c < P.nchunks; c += kCW) {
                const int s = (int)(qc % kLStages);
                if (!__all_sync(kFull, mbar_wait(&bars[s], (uint32_t)(qc / kLStages) & 1, P.err))) {
                    ok = false;
                    break;
                }
                UnitRange R;
                R.lo = (int64_t)c * P.chunk;
                R.hi = min((int64_t)P.V, R.lo + P.chunk);
                R.vlo = R.lo;
                R.nvec = ((R.hi - R.lo) * ES) / 16;
                R.vhi = R.vlo + R.nvec * Elem<DT>::kVec;
                const uint4 *stage = reinterpret_cast<const uint4 *>(slots + (size_t)s * kUnitBytes);
                uint4 v[kVecPerLane];
#pragma unroll
                for (int kk = 0; kk < kVecPerLane; ++kk) {
                    const int vi = kk * 32 + lane;
                    v[kk] = (vi < R.nvec) ? stage[vi] : neg_inf_vec<DT>();
                }
                __syncwarp();
                ++qc;
                if (lane == 0 && ci < P.nchunks) {  // the slot is in registers: refill it
                    issue(row, ci);
                    ci += kCW;
                }
                if (greedy)
                    argmax_regs<DT>(&lpart[c], lane, v, R, row);
                else
                    softmax_regs<DT>(&lpart[c], cs, lane, v, R, row);
            }
            if (!ok && lane == 0)
                *in_block<CS>(&s_abort, 0u) = 1;
            cluster_barrier<CS>();  // the row's chunk partials are in the leader's spart
            if (CS == 1 && s_abort)
                break;
            if constexpr (CUT)
                if (!greedy) {  // uniform: the row's cut key, and its partials over the survivors
                    kl_cut_row<DT>(CutDims{P.V, P.chunk, P.nchunks, P.err, slots}, C, spart,
                                   HOST ? P.lstage + (size_t)(tb + i) * P.lstride * ES : row, cs);
                    if (C.abort)
                        break;  // uniform (read after the cut's last barrier)
                }
            // ---- the row's statistics (K2's per-row combine) and, on a draft row, the test
            if (leader && warp == 0) {
                float m = -INFINITY, sv = 0.f, best = -INFINITY;
                int idx = INT_MAX;
                for (int c = lane; c < P.nchunks; c += 32) {
                    const float2 pc = spart[c];
                    if (greedy) {
                        const int cix = __float_as_int(pc.y);
                        if (pc.x > best || (pc.x == best && cix < idx)) {
                            best = pc.x;
                            idx = cix;
                        }
                    } else if (pc.x != -INFINITY) {
                        const float Mc = pc.x * cs;
                        if (Mc > m) {
                            sv = (m == -INFINITY) ? pc.y : sv * ex2(m - Mc) + pc.y;
                            m = Mc;
                        } else {
                            sv += pc.y * ex2(Mc - m);
                        }
                    }
                }
                bool go = false;
                if (greedy) {
                    warp_argmax(best, idx);
                    am = idx == INT_MAX ? 0 : idx;
                    go = i < k && __shfl_sync(kFull, xs, i) == am;
                } else {
                    const float mw = warp_max(m);
                    const float sw = warp_sum(m == -INFINITY ? 0.f : sv * ex2(m - mw));
                    Mi = mw;
                    Si = sw;
                    bool accept = true;
                    if (lane == i && i < k) {
                        const float e = fmaf(ls, cs, -Mi);
                        const float wstar = kept<DT, CUT>(ls, CUT ? C.thr : 0u) ? ex2(e) : 0.f;
                        const double lhs = (double)ua * (double)qs;  // exact
                        const float ps = wstar / Si;
                        if (ps > 1e-30f || wstar == 0.f)
                            accept = lhs < (double)ps;
                        else  // below fp32's normal range: form p(x*) in double
                            accept = lhs < exp2((double)e) / (double)Si;
                    }
                    go = i < k && __shfl_sync(kFull, accept, i & 31);
                }
                if (lane == 0) {
                    const int g = (CS > 1 && s_abort) ? 2 : (int)go;  // 2: a block gave up on a wait
                    for (unsigned q = 0; q < (unsigned)CS; ++q) {
                        *in_block<CS>(&s_go, q) = g;
                        *in_block<CS>(&s_M, q) = Mi;
                        *in_block<CS>(&s_S, q) = Si;
                    }
                }
            }
            cluster_barrier<CS>();
            if (s_go != 1) {
                j = i;
                break;
            }
        }
        if ((CS == 1 && s_abort) || (CS > 1 && s_go == 2) || (CUT && C.abort))
            break;

        // ---- the output token at row t_j (K2 / K3 arithmetic)
        const int64_t tj = tb + j;
        // rows in host memory: the output row and the draft row come from their device copies
        const char *rowj = (HOST && P.lstage) ? P.lstage + (size_t)tj * P.lstride * ES : row_ptr<DT>(P, tj);
        float *qstage_j = (HOST && P.qstage) ? P.qstage + (db + j) * (int64_t)P.V : nullptr;
        int token = -1;
        bool residual = !greedy && j < k && P.q;
        const uint32_t thr = CUT ? C.thr : 0u;  // cut key of row t_j
        bool drawn = false;
        if constexpr (CUT)
            if (!greedy && C.lok) {  // uniform: row t_j's kept tokens are all listed
                const int mode = j == k ? 2 : (P.q ? 0 : 1);
                // q where it lives (rows in host memory: the device copy is written by the residual
                // pass, which the list makes unnecessary)
                const float *qj = mode == 0 ? P.q + (db + j) * P.qstride : nullptr;
                const int xj = __shfl_sync(kFull, xs, j & 31);
                token = kl_list_draw(C, P.chunk, mode, qj, cs, s_M, 1.f / s_S, xj, __ldg(P.uni + 2 * tj + 1), rowj,
                                     P.V);
                drawn = token >= 0;
                residual = residual && !drawn;
            }
        if (residual) {  // explicit q: residual chunk masses of row t_j by every warp (K3)
            const float Mj = s_M, Sj = s_S;
            const ResidualMass<DT, CUT> f{rowj, P.q + (db + j) * P.qstride, cs, Mj, 1.f / Sj, thr};
            for (int c = cw; c < P.nchunks; c += kCW) {
                const int64_t lo = (int64_t)c * P.chunk, hi = min((int64_t)P.V, (int64_t)(c + 1) * P.chunk);
                const float z = (HOST && qstage_j)
                                    ? warp_residual_chunk<DT, CUT, SPEC_KL_HOST_RESIDUAL_UNROLL, true>(f, lo, hi, lane,
                                                                                                       qstage_j)
                                    : warp_residual_chunk<DT, CUT,
                                                          (DT && !CUT) ? SPEC_KL_RESIDUAL_UNROLL_BF16
                                                                       : SPEC_KL_RESIDUAL_UNROLL>(f, lo, hi, lane);
                if (lane == 0)
                    lrm[c] = z;
            }
            cluster_barrier<CS>();
        }
        if (leader && !drawn) {
            // the draw, by the whole block: chunk masses scanned by every warp alike (smem), the
            // chunk searched by all threads at once (block_find: one round trip to memory)
            const float us = greedy ? 0.f : __ldg(P.uni + 2 * tj + 1);
            if (greedy) {
                token = am;  // warp 0: the argmax of row t_j, the first mismatch or the bonus row
            } else if (j == k) {  // bonus: draw from p
                float M, S;
                warp_combine_soft(spart, P.nchunks, cs, lane, M, S);
                ChunkMassFromPartials cm{spart, cs, M, -1, 0.f};
                const float Z = chunk_total(cm, P.nchunks, lane);
                float th;
                const int c = chunk_locate(cm, P.nchunks, us * Z, lane, th);
                TargetMass<DT, CUT> f{rowj, cs, M, -1, thr};
                token = (int)block_find(f, (int64_t)c * P.chunk, min((int64_t)P.V, (int64_t)(c + 1) * P.chunk), th,
                                        bsearch);
            } else if (!residual) {  // one-hot draft: residual = p without x*
                const float Mj = s_M;
                const int xj = __shfl_sync(kFull, xs, j & 31);
                const int cx = xj / P.chunk;
                TargetMass<DT, CUT> fx{rowj, cs, Mj, xj, thr};
                const float mx = block_range_mass(fx, (int64_t)cx * P.chunk,
                                                  min((int64_t)P.V, (int64_t)(cx + 1) * P.chunk), bsearch);
                ChunkMassFromPartials cm{spart, cs, Mj, cx, mx};
                float Z = chunk_total(cm, P.nchunks, lane);
                int64_t excl = xj;
                if (!(Z > 0.f)) {  // empty residual: draw from p itself
                    cm.override_chunk = -1;
                    Z = chunk_total(cm, P.nchunks, lane);
                    excl = -1;
                }
                float th;
                const int c = chunk_locate(cm, P.nchunks, us * Z, lane, th);
                TargetMass<DT, CUT> f{rowj, cs, Mj, excl, thr};
                token = (int)block_find(f, (int64_t)c * P.chunk, min((int64_t)P.V, (int64_t)(c + 1) * P.chunk), th,
                                        bsearch);
            } else {  // explicit q: locate in the residual (K3)
                const float Mj = s_M, Sj = s_S;
                const ChunkMassFromShared cmz{srm};
                const float Z = chunk_total(cmz, P.nchunks, lane);
                if (Z > 0.f) {
                    float th;
                    const int cc = chunk_locate(cmz, P.nchunks, us * Z, lane, th);
                    const ResidualMass<DT, CUT> f{rowj, qstage_j ? qstage_j : P.q + (db + j) * P.qstride, cs, Mj,
                                                  1.f / Sj, thr};
                    token = (int)block_find(f, (int64_t)cc * P.chunk, min((int64_t)P.V, (int64_t)(cc + 1) * P.chunk),
                                            th, bsearch);
                } else {  // empty residual: draw from p itself
                    const ChunkMassFromPartials cm{spart, cs, Mj, -1, 0.f};
                    const float Zp = chunk_total(cm, P.nchunks, lane);
                    float th;
                    const int cc = chunk_locate(cm, P.nchunks, us * Zp, lane, th);
                    const TargetMass<DT, CUT> ft{rowj, cs, Mj, -1, thr};
                    token = (int)block_find(ft, (int64_t)cc * P.chunk, min((int64_t)P.V, (int64_t)(cc + 1) * P.chunk),
                                            th, bsearch);
                }
            }
        }
        if (leader && warp == 0) {
            // ---- outputs
            if (lane == 0)
                P.out_acc[r] = j;
            for (int i = lane; i <= k; i += 32)
                P.out_tokens[tb + i] = (i < j) ? xs : (i == j ? token : -1);
            if (P.counters) {
                unsigned long long *C = P.counters;
                if (lane == 0) {
                    if (k > 0)
                        atomicAdd(C + SPEC_METRIC_NUM_DRAFTS, 1ull);
                    atomicAdd(C + SPEC_METRIC_NUM_DRAFT_TOKENS, (unsigned long long)k);
                    atomicAdd(C + SPEC_METRIC_NUM_ACCEPTED_TOKENS, (unsigned long long)j);
                    atomicAdd(C + SPEC_METRIC_NUM_VERIFIES, 1ull);
                }
                if (lane < j)
                    atomicAdd(C + SPEC_METRIC_ACCEPTED_PER_POS + lane, 1ull);
            }
        }
        if constexpr (CS == 1)
            __syncthreads();  // spart, srm and the shared scalars are reused by the next request
        // (clusters: the barrier after the next claim orders this request's last reads of
        // them before any write of the next one)
    }
    // gave up on a wait: let this warp's copies still in flight land before exiting
    if (lane == 0)
        for (int64_t q2 = qc; q2 < qi; ++q2)
            mbar_wait(&bars[q2 % kLStages], (uint32_t)(q2 / kLStages) & 1, P.err);
    // a launch chained after another without reading its results still ends after it, so that
    // work the caller queues after this call on the stream waits for both
    if (!P.wait_prior)
        wait_for_prerequisite();
}

// ---------------------------------------------------------------------------------------
// Staging of the draft rows the residual pass reads, when q lives in host memory
// ---------------------------------------------------------------------------------------

// For every request r whose explicit-q recovery is pending (rstate[r] = j >= 0), copies draft
// row d = cu[r] + j of q (host memory, read over the host link) to row d of `stage` (device
// memory, row stride V).  Warps over (request, 16 KB piece) units with eight 16-byte loads in
// flight per lane: one streaming pass over exactly the rows K3 reads.  K3 reading q in place
// interleaves those host loads with its own arithmetic and moves half the bandwidth.
__global__ void __launch_bounds__(kThreads) stage_rows_kernel(Params P, float *stage)
{
    allow_dependents();
    wait_for_prerequisite();  // the decisions
    constexpr int kPiece = 4096;  // floats per unit
    constexpr int kUnroll = 8;
    const int lane = threadIdx.x & 31;
    const int per = (P.V + kPiece - 1) / kPiece;
    const int64_t nunits = (int64_t)P.B * per;
    const bool vec = ((reinterpret_cast<uintptr_t>(P.q) | reinterpret_cast<uintptr_t>(stage)) & 15) == 0 &&
                     (P.qstride & 3) == 0 && (P.V & 3) == 0;
    for (int64_t u = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); u < nunits; u += (int64_t)gridDim.x * kWarps) {
        const int r = (int)(u / per);
        const int c = (int)(u - (int64_t)r * per);
        const int j = P.rstate[r];
        if (j < 0)
            continue;
        const int64_t d = (int64_t)P.cu[r] + j;
        const float *src = P.q + d * P.qstride;
        float *dst = stage + d * (int64_t)P.V;
        const int v0 = c * kPiece, v1 = min(P.V, v0 + kPiece);
        if (vec) {
            for (int v = v0 + 4 * lane; v < v1; v += 4 * 32 * kUnroll) {
                uint4 x[kUnroll];
#pragma unroll
                for (int k = 0; k < kUnroll; ++k)
                    if (v + 128 * k < v1)
                        x[k] = ld_stream(src + v + 128 * k);
#pragma unroll
                for (int k = 0; k < kUnroll; ++k)
                    if (v + 128 * k < v1)
                        *reinterpret_cast<uint4 *>(dst + v + 128 * k) = x[k];
            }
        } else {
            for (int v = v0 + lane; v < v1; v += 32)
                dst[v] = __ldg(src + v);
        }
    }
}

// ---------------------------------------------------------------------------------------
// Acceptance counters (vLLM's spec_decode_* counters, SGLang's accept rate / length)
// ---------------------------------------------------------------------------------------

// counters[SPEC_METRIC_*] += this batch's contributions; requests reported invalid (-1)
// are left out.  Integer sums: the result does not depend on the order of the atomics.
__global__ void __launch_bounds__(kThreads) metrics_kernel(const int32_t *cu, const int32_t *acc, int32_t B,
                                                           unsigned long long *counters)
{
    // Lanes take one request each; every count is summed over the warp first (a ballot's
    // population per accepted position, a warp reduction for the rest), then once per warp into
    // 32-bit block totals, then once per block into the 64-bit counters: integer sums, so the
    // order does not matter.
    __shared__ unsigned s_cnt[SPEC_METRIC_COUNT];
    const int lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < SPEC_METRIC_COUNT; i += blockDim.x)
        s_cnt[i] = 0u;
    __syncthreads();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t r0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); r0 < B; r0 += stride) {
        const int64_t r = r0 + lane;  // warp-uniform loop: every lane takes part in the reductions
        const int a = r < B ? acc[r] : -1;
        const bool valid = a >= 0;
        const int k = valid ? cu[r + 1] - cu[r] : 0;
        const unsigned drafts = __popc(__ballot_sync(kFull, valid && k > 0));
        const unsigned verifies = __popc(__ballot_sync(kFull, valid));
        const unsigned tokens = __reduce_add_sync(kFull, (unsigned)(valid ? k : 0));
        const unsigned accepted = __reduce_add_sync(kFull, (unsigned)(valid ? a : 0));
        const int amax = __reduce_max_sync(kFull, (unsigned)(valid ? a : 0));
        if (lane == 0) {
            if (drafts)
                atomicAdd(&s_cnt[SPEC_METRIC_NUM_DRAFTS], drafts);
            if (verifies)
                atomicAdd(&s_cnt[SPEC_METRIC_NUM_VERIFIES], verifies);
            if (tokens)
                atomicAdd(&s_cnt[SPEC_METRIC_NUM_DRAFT_TOKENS], tokens);
            if (accepted)
                atomicAdd(&s_cnt[SPEC_METRIC_NUM_ACCEPTED_TOKENS], accepted);
        }
        for (int i = 0; i < amax && i < SPEC_REJECT_MAX_SPEC_LEN; ++i) {
            const unsigned n = __popc(__ballot_sync(kFull, valid && a > i));
            if (lane == 0 && n)
                atomicAdd(&s_cnt[SPEC_METRIC_ACCEPTED_PER_POS + i], n);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < SPEC_METRIC_COUNT; i += blockDim.x)
        if (s_cnt[i])
            atomicAdd(counters + i, (unsigned long long)s_cnt[i]);
}

// ---------------------------------------------------------------------------------------
// Greedy tree verification ("投机解码（Speculative Decoding）端到端深挖" §6.2, §7.1)
// ---------------------------------------------------------------------------------------

// One warp per tree.  K1 has left per-chunk (max, argmax) partials for every node row.
// From the root: argmax at the current node; the lowest-index child carrying that token is
// accepted and becomes the current node; otherwise the walk stops and the argmax is the
// bonus.  Invalid trees (node 0 not a root, a parent not preceding its child, a token
// outside the vocabulary) report -1.
__global__ void __launch_bounds__(kThreads) tree_walk_kernel(Params P, const int32_t *parent, const int32_t *tok,
                                                             const int32_t *cu_nodes, int32_t B, int32_t *out_tokens,
                                                             int32_t *out_acc, int32_t *out_last)
{
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (r >= B)
        return;
    const int n0 = cu_nodes[r];
    const int n = cu_nodes[r + 1] - n0;
    bool bad = n < 1 || n0 < 0 || (int64_t)n0 + n > P.T;
    if (!bad) {
        bool lbad = false;
        for (int i = lane; i < n; i += 32) {
            const int pi = parent[n0 + i];
            lbad |= (i == 0) ? pi != -1 : (pi < 0 || pi >= i || tok[n0 + i] < 0 || tok[n0 + i] >= P.V);
        }
        bad = __any_sync(kFull, lbad);
    }
    if (bad) {
        if (n >= 1 && n0 >= 0 && (int64_t)n0 + n <= P.T)
            for (int i = lane; i < n; i += 32)
                out_tokens[n0 + i] = -1;
        if (lane == 0) {
            out_acc[r] = -1;
            out_last[r] = -1;
            atomicOr(P.err, SPEC_DEVERR_TREE);
            atomicMin(P.err + 1, r);
        }
        return;
    }
    int cur = 0, acc = 0;
    for (int step = 0; step < n; ++step) {
        const int am = warp_combine_argmax(P.part + ((int64_t)n0 + cur) * P.nchunks, P.nchunks, lane);
        int child = INT_MAX;
        for (int i = 1 + lane; i < n; i += 32)
            if (parent[n0 + i] == cur && tok[n0 + i] == am)
                child = min(child, i);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            child = min(child, __shfl_xor_sync(kFull, child, o));
        if (lane == 0)
            out_tokens[n0 + acc] = am;
        if (child == INT_MAX)
            break;
        ++acc;
        cur = child;
    }
    for (int i = acc + 1 + lane; i < n; i += 32)
        out_tokens[n0 + i] = -1;
    if (lane == 0) {
        out_acc[r] = acc;
        out_last[r] = cur;
    }
}

// ---------------------------------------------------------------------------------------
// n-gram draft proposer ("第12章 投机解码：以小博大" §12.4.4)
// ---------------------------------------------------------------------------------------

// One block per request, one pass over its context for every n at once: each thread takes
// candidate starts s (SPEC_NGRAM_PER at a time, their first tokens loaded together), and at each s
// finds the largest n in [min_n, max_n] whose last n context tokens occur at s wholly before
// the final n tokens (s <= L - 2n); a first-token test against the n suffixes, held in shared
// memory, settles almost every s.  The block keeps the best (n, then the smallest s) as one
// 64-bit key (n above, 2^40 - 1 - s below) reduced by a maximum; the proposal is the (at most
// k) tokens after that occurrence.
#ifndef SPEC_NGRAM_PER
#define SPEC_NGRAM_PER 4  // candidate starts per thread per sweep
#endif
#ifndef SPEC_NGRAM_MIN_BLOCKS
#define SPEC_NGRAM_MIN_BLOCKS 8  // resident blocks per SM the registers must allow (one wave at B = 1024)
#endif
constexpr int kNgramPer = SPEC_NGRAM_PER;
__global__ void __launch_bounds__(kThreads, SPEC_NGRAM_MIN_BLOCKS) ngram_kernel(const int32_t *tokens, const int64_t *cu, int32_t B,
                                                         int min_n, int max_n, int k, int64_t max_model_len,
                                                         int32_t *out, int32_t *out_num)
{
    constexpr unsigned long long kSMask = (1ull << 40) - 1;
    __shared__ int32_t suf[SPEC_NGRAM_MAX_N];  // the last nmax tokens of the context
    __shared__ unsigned long long s_best[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = blockIdx.x; r < B; r += gridDim.x) {
        const int64_t c0 = cu[r];
        const int64_t L = cu[r + 1] - c0;
        const int32_t *ctx = tokens + c0;
        int64_t kk = k;
        if (max_model_len > 0)
            kk = min(kk, max_model_len - L);
        const int nmax = (int)min((int64_t)max_n, L / 2);  // 2n <= L
        const bool search = kk > 0 && nmax >= min_n;
        __syncthreads();  // suf and s_best of the previous request are no longer read
        if (search && (int)threadIdx.x < nmax)
            suf[threadIdx.x] = ctx[L - nmax + threadIdx.x];
        __syncthreads();
        unsigned long long best = 0;
        if (search) {
            const int64_t last = L - 2 * (int64_t)min_n;  // the largest start for the shortest n
            const int64_t step = (int64_t)blockDim.x * kNgramPer;
            for (int64_t s0 = 0; s0 <= last; s0 += step) {
                int32_t t0[kNgramPer];
#pragma unroll
                for (int u = 0; u < kNgramPer; ++u) {
                    const int64_t st = s0 + (int64_t)u * blockDim.x + threadIdx.x;
                    t0[u] = st <= last ? ctx[st] : 0;
                }
#pragma unroll
                for (int u = 0; u < kNgramPer; ++u) {
                    const int64_t st = s0 + (int64_t)u * blockDim.x + threadIdx.x;
                    if (st > last)
                        continue;
                    for (int n = (int)min((int64_t)nmax, (L - st) / 2); n >= min_n; --n) {
                        const int32_t *pat = suf + (nmax - n);  // the last n tokens
                        if (t0[u] != pat[0])
                            continue;
                        bool ok = true;
                        for (int i = 1; ok && i < n; ++i)
                            ok = ctx[st + i] == pat[i];
                        if (ok) {
                            best = max(best, ((unsigned long long)n << 40) | (kSMask - (unsigned long long)st));
                            break;  // the largest n at this start
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            best = max(best, __shfl_xor_sync(kFull, best, o));
        if (lane == 0)
            s_best[warp] = best;
        __syncthreads();
        best = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w)
            best = max(best, s_best[w]);
        const int found_n = (int)(best >> 40);
        const int64_t found = best ? (int64_t)(kSMask - (best & kSMask)) : -1;
        const int cnt = found < 0 ? 0 : (int)min(kk, L - (found + found_n));
        for (int i = threadIdx.x; i < k; i += blockDim.x)
            out[(int64_t)r * k + i] = i < cnt ? ctx[found + found_n + i] : -1;
        if (threadIdx.x == 0)
            out_num[r] = cnt;
    }
}

// ---------------------------------------------------------------------------------------
// Diagnostics: per-row statistics from K1's partials
// ---------------------------------------------------------------------------------------

// One warp per row: m_t and s_t = sum exp((l - m_t) / T_r) (sampling rows, x* included).
template <int DT>
__global__ void __launch_bounds__(kThreads) debug_soft_kernel(Params P, float *row_max, float *row_sum)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= P.T || P.B == 0 || (P.err[0] & SPEC_DEVERR_LAYOUT))
        return;
    const int r = find_request(P, t);
    const float temp = P.temp[r];
    if (!(temp > 0.f))
        return;  // greedy rows: filled from the argmax pass
    const float cs = kLog2e / temp;
    float M, S;
    warp_combine_soft(P.part + t * P.nchunks, P.nchunks, cs, lane, M, S);
    float m = -INFINITY;
    for (int c = lane; c < P.nchunks; c += 32)
        m = fmaxf(m, P.part[t * P.nchunks + c].x);
    m = warp_max(m);
    if (lane == 0) {
        if (row_max)
            row_max[t] = m;
        if (row_sum)  // S is relative to 2^M; rescale to exp(-m / T)
            row_sum[t] = (float)((double)S * exp2((double)M - (double)m * (double)cs));
    }
}

// One warp per row after an argmax pass: lowest-index argmax (and the max on greedy rows).
__global__ void __launch_bounds__(kThreads) debug_argmax_kernel(Params P, float *row_max, float *row_sum,
                                                                int32_t *row_argmax)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= P.T || P.B == 0 || (P.err[0] & SPEC_DEVERR_LAYOUT))
        return;
    const int idx = warp_combine_argmax(P.part + t * P.nchunks, P.nchunks, lane);
    if (lane == 0) {
        if (row_argmax)
            row_argmax[t] = idx;
        const int r = find_request(P, t);
        if (!(P.temp[r] > 0.f)) {
            float best;
            lane_combine_argmax(P, t, &best);
            if (row_max)
                row_max[t] = best;
            if (row_sum)
                row_sum[t] = 0.f;
            const int64_t i = t - ((int64_t)P.cu[r] + r);
            if (P.dbg_pdraft && i < P.cu[r + 1] - P.cu[r])
                P.dbg_pdraft[t - r] = 0.f;
        }
    }
}

#ifdef SPEC_KL_CUT_VARIANT
// ---------------------------------------------------------------------------------------
// This file compiled a second time (spec_reject_cut16.cu) with kLWarps = 16: the first-
// rejection pass with cuts, one 16-warp block per SM.  Only its launcher and occupancy query
// are visible to the other translation unit; everything else here has internal linkage.
// ---------------------------------------------------------------------------------------
}  // namespace

// Blocks of the 16-warp pass with cuts that fit on one SM (0: none), after raising its
// dynamic shared-memory limit.
cudaError_t lazy_cut16_blocks_per_sm(int *blocks)
{
    cudaError_t e = cudaFuncSetAttribute(lazy_kernel<1, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kLCutSmem);
    if (e != cudaSuccess)
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, lazy_kernel<1, false, true>, kLThreads, kLCutSmem);
}

// Launch of the 16-warp pass with cuts (rows in device memory), with `pdl` as a programmatic
// dependent launch of the layout check.
cudaError_t launch_lazy_cut16(const Params &P, int grid, bool pdl, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kLThreads, 1, 1);
    cfg.dynamicSmemBytes = kLCutSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, lazy_kernel<1, false, true>, P);
}
}  // namespace specrej
#else
}  // namespace
// The 16-warp pass with cuts, from the second translation unit of this file.
cudaError_t lazy_cut16_blocks_per_sm(int *blocks);
cudaError_t launch_lazy_cut16(const Params &P, int grid, bool pdl, cudaStream_t stream);
namespace {

// ---------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------

struct DeviceInfo {
    int sms = 0;
    int blocks_rowstats[2] = {0, 0};
    int blocks_residual[2] = {0, 0};
    int blocks_wr[2] = {0, 0};
    int blocks_lazy[2] = {0, 0};
    int blocks_lazy_cut = 0;       // KL with cuts (bf16)
    int blocks_lazy_cut16 = 0;     // the same with 16-warp blocks (spec_reject_cut16.cu)
    int blocks_lazy_cut_host = 0;  // the same, rows in host memory
    int clusters_lazy[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};  // KL with clusters of 1, 2, 4, 8 blocks
};

constexpr size_t kWrSmem = (size_t)kWrWarps * kWrStages * kUnitBytes;

constexpr int kMaxDevices = 64;
// Per-device launch-shape cache (SM count, occupancy), filled once per device by the first
// call made with that device current; std::call_once makes concurrent first calls from
// several host threads safe (the others wait for the fill, then read it).
DeviceInfo g_dev[kMaxDevices];
cudaError_t g_dev_err[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

// Launch of KL with clusters of CS blocks (CS > 1): one cluster per request at a time.
// Launch of KL (any variant; clusters of CS blocks when CS > 1), after the layout check: with
// `pdl` as a programmatic dependent launch (the kernel waits for the check's writes itself).
template <class K>
cudaError_t launch_lazy(K kernel, int grid, int cs, size_t smem, const Params &P, bool pdl, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kLThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cs > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cs;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, P);
}

// Launch of a kernel of the full pass, as a programmatic dependent launch of the kernel before it
// on the stream when `pdl` (the kernel waits for that one's writes itself).
template <class... A, class... B>
cudaError_t launch_dep(void (*kernel)(A...), int grid, int block, size_t smem, bool pdl, cudaStream_t stream,
                       B... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int DT, int CS> cudaError_t launch_lazy_cluster(const Params &P, int clusters, bool pdl, cudaStream_t stream)
{
    return launch_lazy(lazy_kernel<DT, false, false, CS>, clusters * CS, CS, kLSmem, P, pdl, stream);
}

// Clusters of CS blocks of KL that fit on the device at once (whole GPU).
template <int DT, int CS> cudaError_t lazy_cluster_occupancy(int &clusters)
{
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(lazy_kernel<DT, false, false, CS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kLSmem)))
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(CS * 64), 1, 1);
    cfg.blockDim = dim3(kLThreads, 1, 1);
    cfg.dynamicSmemBytes = kLSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&clusters, lazy_kernel<DT, false, false, CS>, &cfg);
    if (e) {  // clusters of this size cannot run here: the call keeps to smaller ones
        (void)cudaGetLastError();
        clusters = 0;
        return cudaSuccess;
    }
    return cudaSuccess;
}

template <int DT> cudaError_t fill_info(DeviceInfo &di)
{
    cudaError_t e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&di.blocks_rowstats[DT], rowstats_kernel<DT>, kThreads, 0)))
        return e;
    if ((e = cudaFuncSetAttribute(rowstats_wr_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWrSmem)))
        return e;
    // two cut blocks per SM: one block's loads overlap the other's selection
    if ((e = cudaFuncSetAttribute(filter_kernel<DT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)))
        return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&di.blocks_wr[DT], rowstats_wr_kernel<DT>, kWrThreads,
                                                           kWrSmem)))
        return e;
    if ((e = cudaFuncSetAttribute(lazy_kernel<DT, false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kLSmem)))
        return e;
    if ((e = cudaFuncSetAttribute(lazy_kernel<DT, true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kLSmem)))
        return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&di.blocks_lazy[DT], lazy_kernel<DT, false, false>,
                                                           kLThreads, kLSmem)))
        return e;
    if ((e = lazy_cluster_occupancy<DT, 2>(di.clusters_lazy[DT][1])) || (e = lazy_cluster_occupancy<DT, 4>(di.clusters_lazy[DT][2])) ||
        (e = lazy_cluster_occupancy<DT, 8>(di.clusters_lazy[DT][3])))
        return e;
    di.clusters_lazy[DT][0] = di.blocks_lazy[DT];  // per SM; multiplied by the SM count at launch
    if constexpr (DT == 1) {
        if ((e = cudaFuncSetAttribute(lazy_kernel<1, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kLCutSmem)))
            return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&di.blocks_lazy_cut, lazy_kernel<1, false, true>,
                                                               kLThreads, kLCutSmem)))
            return e;
        if ((e = cudaFuncSetAttribute(lazy_kernel<1, true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kLCutSmem)))
            return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&di.blocks_lazy_cut_host, lazy_kernel<1, true, true>,
                                                               kLThreads, kLCutSmem)))
            return e;
        if ((e = lazy_cut16_blocks_per_sm(&di.blocks_lazy_cut16)))
            return e;
    }
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&di.blocks_residual[DT], residual_kernel<DT, false>, kThreads, 0);
}

cudaError_t device_info(DeviceInfo **out)
{
    int dev;
    cudaError_t e = cudaGetDevice(&dev);
    if (e)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::call_once(g_dev_once[dev], [dev]() {
        DeviceInfo tmp;
        cudaError_t e2 = cudaDeviceGetAttribute(&tmp.sms, cudaDevAttrMultiProcessorCount, dev);
        if (!e2)
            e2 = fill_info<0>(tmp);
        if (!e2)
            e2 = fill_info<1>(tmp);
        if (!e2)
            g_dev[dev] = tmp;
        g_dev_err[dev] = e2;
    });
    if (g_dev_err[dev])
        return g_dev_err[dev];
    *out = &g_dev[dev];
    return cudaSuccess;
}

// A CUDA error that earlier work left pending on the calling thread (cudaPeekAtLastError) is
// not this call's: the entry points report it as SPEC_ERR_CUDA before launching anything and
// leave it pending, so that the launch checks after their own launches see only their own.
bool cuda_error_pending() { return cudaPeekAtLastError() != cudaSuccess; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// log2 of the blocks per request of KL on device rows without cuts: clusters serve batches too
// small to fill the GPU one block per request.  The largest cluster (at most 8 blocks) such
// that the GPU holds a cluster for every request at once and every warp of a cluster has at
// least one chunk of each row (a cluster serialises its requests' draws, and its barriers cost
// more than a small row saves).
// Requests of a batch that fills the GPU one block per request that are served by a second
// launch with two blocks per request (see run()): a share of the blocks the first launch holds,
// for batches of at least three times that many requests whose rows give each warp of a pair a
// chunk; 0 otherwise.
#ifndef SPEC_KL_CUT16_PER_SM
#define SPEC_KL_CUT16_PER_SM 4  // requests per SM up to which the pass with cuts runs 16-warp blocks
#endif

#ifndef SPEC_KL_CUT_TAIL_PERMILLE
#define SPEC_KL_CUT_TAIL_PERMILLE 1000  // requests per 1000 SMs run by the 16-warp build after a large batch's cut pass
#endif

#ifndef SPEC_KL_TAIL_PERMILLE
#define SPEC_KL_TAIL_PERMILLE 300  // tail requests per 1000 blocks of the first launch
#endif
int lazy_tail_requests(const DeviceInfo &di, int DT, int32_t B, int nchunks)
{
    const int64_t blocks = (int64_t)di.sms * di.blocks_lazy[DT];
    const int64_t tail = blocks * SPEC_KL_TAIL_PERMILLE / 1000;
    if (tail < 1 || di.clusters_lazy[DT][1] <= 0 || (kLWarps << 1) > nchunks || (int64_t)B < 3 * tail + blocks)
        return 0;
    return (int)tail;
}

// Requests of a batch with cuts on device rows that the 16-warp build of the pass takes: all of
// them for batches of at most SPEC_KL_CUT16_PER_SM requests per SM, else the last
// SPEC_KL_CUT_TAIL_PERMILLE per 1000 SMs, in a second launch chained to the 8-warp one; 0
// without that build.
int64_t lazy_cut16_requests(const DeviceInfo &di, int32_t B)
{
    if (di.blocks_lazy_cut16 <= 0)
        return 0;
    if ((int64_t)B <= (int64_t)di.sms * SPEC_KL_CUT16_PER_SM)
        return B;
    return (int64_t)di.sms * SPEC_KL_CUT_TAIL_PERMILLE / 1000;
}

int lazy_cluster_log2(const DeviceInfo &di, int DT, int32_t B, int nchunks)
{
    if (SPEC_KL_CLUSTER_LOG2 >= 0)
        return di.clusters_lazy[DT][SPEC_KL_CLUSTER_LOG2] > 0 ? SPEC_KL_CLUSTER_LOG2 : 0;
    for (int c = 3; c >= 1; --c)
        if (di.clusters_lazy[DT][c] >= B && (kLWarps << c) <= nchunks)
            return c;
    return 0;
}

// Blocks for a persistent launch: enough to fill every SM at full occupancy, no more
// than there is work for, at least one.
int64_t clamp_grid(int64_t full, int64_t needed)
{
    const int64_t g = needed < full ? needed : full;
    return g < 1 ? 1 : g;
}

spec_status check_args(const void *logits, spec_dtype dt, int64_t T, int32_t V, int64_t lstride, const float *q,
                       int64_t qstride, const int32_t *ids, const int32_t *cu, int32_t B, const float *uni,
                       const float *temp, int32_t *out_tokens, int32_t *out_acc, void *ws)
{
    if (dt != SPEC_F32 && dt != SPEC_BF16)
        return SPEC_ERR_INVALID_ARG;
    if (B < 0 || T < 0 || V < 1 || T < B)
        return SPEC_ERR_INVALID_ARG;
    if (V > SPEC_REJECT_MAX_VOCAB)
        return SPEC_ERR_UNSUPPORTED;
    if (lstride != 0 && lstride < V)
        return SPEC_ERR_INVALID_ARG;
    if (q && qstride != 0 && qstride < V)
        return SPEC_ERR_INVALID_ARG;
    if (!cu || !ws || (T > 0 && (!logits || !uni || !out_tokens)) || (B > 0 && (!temp || !out_acc)) ||
        (T > B && !ids))
        return SPEC_ERR_INVALID_ARG;
    const size_t es = dt == SPEC_BF16 ? 2 : 4;
    if (!aligned(logits, es) || !aligned(q, 4) || !aligned(ids, 4) || !aligned(cu, 4) || !aligned(uni, 4) ||
        !aligned(temp, 4) || !aligned(out_tokens, 4) || !aligned(out_acc, 4))
        return SPEC_ERR_INVALID_ARG;
    return SPEC_OK;
}

// K1: the TMA ring when every row starts on a 16-byte boundary (the common case), the
// register-staged kernel otherwise.
void launch_rowstats(int DT, const Params &P, const DeviceInfo &di, int64_t T, int nchunks, const void *logits,
                     int64_t lstride, int gridA, cudaStream_t stream, int force_argmax)
{
    const size_t es = DT ? 2 : 4;
    const bool rows_aligned = aligned(logits, 16) && ((size_t)lstride * es) % 16 == 0;
    if (rows_aligned && di.blocks_wr[DT] > 0) {
        const int64_t units = T * (int64_t)nchunks;
        const int64_t warps_needed = (units + 3) / 4;  // at least ~4 units per warp
        const int grid = (int)clamp_grid((int64_t)di.sms * di.blocks_wr[DT], (warps_needed + kWrWarps - 1) / kWrWarps);
        if (DT)
            rowstats_wr_kernel<1><<<grid, kWrThreads, kWrSmem, stream>>>(P, force_argmax);
        else
            rowstats_wr_kernel<0><<<grid, kWrThreads, kWrSmem, stream>>>(P, force_argmax);
    } else {
        if (DT)
            rowstats_kernel<1><<<gridA, kThreads, 0, stream>>>(P, force_argmax);
        else
            rowstats_kernel<0><<<gridA, kThreads, 0, stream>>>(P, force_argmax);
    }
}

// K1F: one cluster per target row (blocks of unfiltered rows exit at once).
cudaError_t launch_filter(int DT, const Params &P, int64_t T, int nchunks, cudaStream_t stream, bool pdl)
{
    const int csize = (nchunks + kFilterMaxChunksPerBlock - 1) / kFilterMaxChunksPerBlock;
    const int cpc = (nchunks + csize - 1) / csize;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(T * csize), 1, 1);
    cfg.blockDim = dim3(kFilterThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    (void)cpc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return DT ? cudaLaunchKernelEx(&cfg, filter_kernel<1>, P, csize) : cudaLaunchKernelEx(&cfg, filter_kernel<0>, P, csize);
}

spec_status run(const void *logits, spec_dtype dt, int64_t T, int32_t V, int64_t lstride, const float *q,
                int64_t qstride, const int32_t *ids, const int32_t *cu, int32_t B, const float *uni,
                const float *temp, int32_t *out_tokens, int32_t *out_acc, void *ws, size_t ws_bytes,
                cudaStream_t stream, float *dbg_m, float *dbg_s, int32_t *dbg_am, float *dbg_pd, float *dbg_z,
                cudaEvent_t *ev = nullptr, int nev = 0, const int32_t *top_k = nullptr, const float *top_p = nullptr,
                int64_t *counters = nullptr, float *q_stage = nullptr, bool rows_in_host = false,
                char *row_stage = nullptr)
{
    spec_status st = check_args(logits, dt, T, V, lstride, q, qstride, ids, cu, B, uni, temp, out_tokens, out_acc, ws);
    if (st != SPEC_OK)
        return st;
    Plan pl;
    if (!make_plan(B, T, V, dt, q != nullptr, &pl))
        return SPEC_ERR_INVALID_ARG;
    if (ws_bytes < pl.total)
        return SPEC_ERR_WORKSPACE;
    DeviceInfo *di;
    if (cuda_error_pending() || device_info(&di) != cudaSuccess)
        return SPEC_ERR_CUDA;

    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
    Params P{};  // every optional pointer starts null
    P.logits = logits;
    P.T = T;
    P.V = V;
    P.lstride = lstride;
    P.q = q;
    P.qstride = qstride;
    P.ids = ids;
    P.cu = cu;
    P.B = B;
    P.uni = uni;
    P.temp = temp;
    P.out_tokens = out_tokens;
    P.out_acc = out_acc;
    P.part = reinterpret_cast<float2 *>(base + pl.off_part);
    P.err = reinterpret_cast<int32_t *>(base + pl.off_err);
    P.rstate = q ? reinterpret_cast<int32_t *>(base + pl.off_rstate) : nullptr;
    P.rstat = reinterpret_cast<float2 *>(base + pl.off_rstat);
    P.rpart = q ? reinterpret_cast<float *>(base + pl.off_rpart) : nullptr;
    P.rcnt = q ? reinterpret_cast<int32_t *>(base + pl.off_rcnt) : nullptr;
    P.chunk = pl.chunk;
    P.nchunks = pl.nchunks;
    P.dbg_pdraft = dbg_pd;
    if (counters && !aligned(counters, 8))
        return SPEC_ERR_INVALID_ARG;
    P.counters = reinterpret_cast<unsigned long long *>(counters);
    P.dbg_z = dbg_z;
    P.r_begin = 0;
    P.r_end = B;
    P.qslot = 2;
    P.wait_prior = 1;
    const bool filtered = top_k || top_p;
    if (filtered) {
        if (!aligned(top_k, 4) || !aligned(top_p, 4) ||
            (pl.nchunks + kFilterMaxChunksPerBlock - 1) / kFilterMaxChunksPerBlock > kFilterMaxCluster)
            return pl.nchunks > kFilterMaxChunksPerBlock * kFilterMaxCluster ? SPEC_ERR_UNSUPPORTED
                                                                            : SPEC_ERR_INVALID_ARG;
        P.top_k = top_k;
        P.top_p = top_p;
        P.thr = reinterpret_cast<uint32_t *>(base + pl.off_thr);
    }

    const int DT = dt == SPEC_BF16 ? 1 : 0;
    const int64_t units = T * (int64_t)pl.nchunks;
    const int64_t full = (int64_t)di->sms * (di->blocks_rowstats[DT] > 0 ? di->blocks_rowstats[DT] : 1);
    const int gridA = (int)clamp_grid(full, (units + kWarps - 1) / kWarps);
    const int gridB = (int)((B + kWarps - 1) / kWarps);
    const bool debug = dbg_m || dbg_s || dbg_am || dbg_pd || dbg_z;

    // stage events: [0] before K1, then one after each kernel launched: K1, K1F (filtered
    // calls only), K2, K3 (explicit draft probabilities only)
    int evi = 0;
    bool marked = false;  // the latest mark() recorded an event (the next launch then is no dependent launch)
    auto mark = [&]() {
        marked = evi < nev && ev[evi];
        if (marked)
            cudaEventRecord(ev[evi], stream);
        ++evi;
    };
    // calls without diagnostics (and with cuts only on bf16 rows, which in host memory need a
    // device copy to cut from): KL reads rows only up to each request's first rejection
    const bool rows_aligned = aligned(logits, 16) && ((size_t)lstride * (DT ? 2 : 4)) % 16 == 0;
    const bool cut_ok = !filtered || (DT == 1 && (rows_in_host ? row_stage && di->blocks_lazy_cut_host > 0
                                                               : di->blocks_lazy_cut > 0));
    // any B >= 1 on device rows without cuts (small batches in clusters of blocks); with cuts,
    // or rows in host memory, batches of at least SPEC_KL_MIN_REQUESTS
    const bool kl_batch = B >= ((filtered || rows_in_host) ? SPEC_KL_MIN_REQUESTS : 1);
    if (cut_ok && !debug && (!q_stage || rows_in_host) && kl_batch && T > 0 && rows_aligned &&
        di->blocks_lazy[DT] > 0) {
        mark();
        lazy_init_kernel<<<1, 256, 0, stream>>>(P);
        // the pass follows as a programmatic dependent launch unless a stage event separates them
        const bool pdl = !(evi < nev && ev[evi]);
        mark();
        if (rows_in_host) {
            // the rows it reads over the host link are copied to device memory for the cut, the
            // residual pass and the draw (q_stage: rows of V floats, row_stage: rows of lstride)
            P.lstage = row_stage;
            P.qstage = q ? q_stage : nullptr;
        }
        if (filtered) {
            // small batches: 16-warp blocks, one per SM, which cut each reached row twice as fast
            // (a row's cut takes most of its time, bound by instruction issue inside the block)
            const int64_t n16 = rows_in_host ? 0 : lazy_cut16_requests(*di, B);
            const bool w16 = n16 == (int64_t)B;
            const int gridL = (int)clamp_grid(
                (int64_t)di->sms * (rows_in_host ? di->blocks_lazy_cut_host
                                                 : (w16 ? di->blocks_lazy_cut16 : di->blocks_lazy_cut)), B);
            // larger batches: 8-warp blocks (two per SM), except the last requests, which run in a
            // second launch of the 16-warp build chained to the first: its blocks take SMs as the
            // first launch's blocks run out of requests, and finish their chains faster
            const int64_t tail16 = w16 ? 0 : n16;
            Params Pm = P;
            Pm.r_end = (int32_t)(B - tail16);
            cudaError_t e = rows_in_host ? launch_lazy(lazy_kernel<1, true, true>, gridL, 1, kLCutSmem, P, pdl, stream)
                            : w16        ? launch_lazy_cut16(P, gridL, pdl, stream)
                                         : launch_lazy(lazy_kernel<1, false, true>, gridL, 1, kLCutSmem, Pm, pdl, stream);
            if (e == cudaSuccess && tail16 > 0) {
                Params Pt = P;
                Pt.r_begin = (int32_t)(B - tail16);
                Pt.qslot = 3;
                Pt.wait_prior = 0;
                e = launch_lazy_cut16(Pt, (int)clamp_grid((int64_t)di->sms * di->blocks_lazy_cut16, tail16), true,
                                      stream);
            }
            mark();
            return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
        }
        const int gridL = (int)clamp_grid((int64_t)di->sms * di->blocks_lazy[DT], B);
        if (!rows_in_host) {
            // clusters of CS blocks per request, for batches too small to fill the GPU one block per
            // request: the largest CS (at most 8) such that the GPU holds a cluster for every request
            // at once and every warp of a cluster has at least one chunk of each row (a cluster
            // serialises its requests' draws, and its barriers cost more than a small row saves)
            const int ci = lazy_cluster_log2(*di, DT, B, pl.nchunks);
            if (ci > 0) {
                const int ncl = (int)clamp_grid(di->clusters_lazy[DT][ci], B);
                cudaError_t e;
                if (DT)
                    e = ci == 1 ? launch_lazy_cluster<1, 2>(P, ncl, pdl, stream)
                                : ci == 2 ? launch_lazy_cluster<1, 4>(P, ncl, pdl, stream)
                                          : launch_lazy_cluster<1, 8>(P, ncl, pdl, stream);
                else
                    e = ci == 1 ? launch_lazy_cluster<0, 2>(P, ncl, pdl, stream)
                                : ci == 2 ? launch_lazy_cluster<0, 4>(P, ncl, pdl, stream)
                                          : launch_lazy_cluster<0, 8>(P, ncl, pdl, stream);
                mark();
                return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
            }
        }
        const int tail = rows_in_host ? 0 : lazy_tail_requests(*di, DT, B, pl.nchunks);
        Params Pm = P;
        Pm.r_end = B - tail;
        cudaError_t e;
        if (rows_in_host)
            e = DT ? launch_lazy(lazy_kernel<1, true, false>, gridL, 1, kLSmem, Pm, pdl, stream)
                   : launch_lazy(lazy_kernel<0, true, false>, gridL, 1, kLSmem, Pm, pdl, stream);
        else
            e = DT ? launch_lazy(lazy_kernel<1, false, false>, gridL, 1, kLSmem, Pm, pdl, stream)
                   : launch_lazy(lazy_kernel<0, false, false>, gridL, 1, kLSmem, Pm, pdl, stream);
        if (e == cudaSuccess && tail > 0) {
            // the last requests, two blocks each, in a launch chained after the first (it reads
            // none of the first's results): its clusters take SM slots as the first launch's
            // blocks run out of requests, and finish their requests twice as fast
            Params Pt = P;
            Pt.r_begin = B - tail;
            Pt.qslot = 3;
            Pt.wait_prior = 0;
            const int ncl = (int)clamp_grid(di->clusters_lazy[DT][1], tail);
            e = DT ? launch_lazy_cluster<1, 2>(Pt, ncl, true, stream) : launch_lazy_cluster<0, 2>(Pt, ncl, true, stream);
        }
        mark();
        return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
    }
    if (rows_in_host)
        return SPEC_ERR_INVALID_ARG;  // only the first-rejection pass reads rows in host memory
    // the full pass: K1, then K1F / K2 / K3 each as a programmatic dependent launch of the kernel
    // before it (no stage event between them)
    mark();
    launch_rowstats(DT, P, *di, T, pl.nchunks, logits, lstride, gridA, stream, 0);
    mark();
    bool chain = true;  // the kernel just launched is one of the pass's (a debug kernel is not)
    if (filtered && T > 0 && B > 0) {
        if (launch_filter(DT, P, T, pl.nchunks, stream, chain && !marked) != cudaSuccess)
            return SPEC_ERR_CUDA;
        mark();
    }
    if (debug && T > 0 && (dbg_m || dbg_s)) {
        const int g = (int)((T + kWarps - 1) / kWarps);
        if (DT)
            debug_soft_kernel<1><<<g, kThreads, 0, stream>>>(P, dbg_m, dbg_s);
        else
            debug_soft_kernel<0><<<g, kThreads, 0, stream>>>(P, dbg_m, dbg_s);
        chain = false;
    }
    if (B > 0) {
        const bool F = P.thr != nullptr;
        cudaError_t e = DT ? launch_dep(F ? finalize_kernel<1, true> : finalize_kernel<1, false>, gridB, kThreads, 0,
                                        chain && !marked, stream, P)
                           : launch_dep(F ? finalize_kernel<0, true> : finalize_kernel<0, false>, gridB, kThreads, 0,
                                        chain && !marked, stream, P);
        if (e != cudaSuccess)
            return SPEC_ERR_CUDA;
        mark();
        if (q) {
            Params P3 = P;
            if (q_stage) {  // q in host memory: stage the rows K3 reads into device memory first
                const int64_t sunits = (int64_t)B * ((V + 4095) / 4096);
                const int gridS = (int)clamp_grid((int64_t)di->sms * 8, (sunits + kWarps - 1) / kWarps);
                if (launch_dep(stage_rows_kernel, gridS, kThreads, 0, !marked, stream, P, q_stage) != cudaSuccess)
                    return SPEC_ERR_CUDA;
                P3.q = q_stage;
                P3.qstride = V;
            }
            const int64_t runits = (int64_t)B * pl.nchunks;
            const int64_t rfull = (int64_t)di->sms * (di->blocks_residual[DT] > 0 ? di->blocks_residual[DT] : 1);
            const int gridC = (int)clamp_grid(rfull, (runits + kWarps - 1) / kWarps);
            const bool pdl3 = q_stage ? true : !marked;  // after the staging kernel, or after K2
            e = DT ? launch_dep(F ? residual_kernel<1, true> : residual_kernel<1, false>, gridC, kThreads, 0, pdl3,
                                stream, P3)
                   : launch_dep(F ? residual_kernel<0, true> : residual_kernel<0, false>, gridC, kThreads, 0, pdl3,
                                stream, P3);
            if (e != cudaSuccess)
                return SPEC_ERR_CUDA;
            mark();
        }
    }
    if (debug && T > 0 && B > 0 && (dbg_am || dbg_m || dbg_s || dbg_pd)) {
        // argmax of every row (the sampling path does not need it), then per-row combine
        launch_rowstats(DT, P, *di, T, pl.nchunks, logits, lstride, gridA, stream, kArgmaxKeepErrors);
        const int g = (int)((T + kWarps - 1) / kWarps);
        debug_argmax_kernel<<<g, kThreads, 0, stream>>>(P, dbg_m, dbg_s, dbg_am);
    }
    if (cudaGetLastError() != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

}  // namespace
}  // namespace specrej

using namespace specrej;

// ---------------------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------------------

extern "C" {

size_t spec_reject_workspace_size(int32_t B, int64_t T, int32_t V, spec_dtype logits_dtype, int has_draft_probs)
{
    Plan pl;
    if (!make_plan(B, T, V, logits_dtype, has_draft_probs, &pl))
        return 0;
    return pl.total;
}

spec_status spec_reject_sample(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                               int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                               const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                               const float *uniforms, const float *temperature, int32_t *out_tokens,
                               int32_t *out_num_accepted, void *workspace, size_t workspace_bytes, void *stream)
{
    return run(target_logits, logits_dtype, T, V, logits_row_stride, draft_probs, q_row_stride, draft_ids,
               cu_num_draft, B, uniforms, temperature, out_tokens, out_num_accepted, workspace, workspace_bytes,
               static_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr, nullptr, nullptr);
}

spec_status spec_reject_sample_filtered(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                        int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                        const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                        const float *uniforms, const float *temperature, const int32_t *top_k,
                                        const float *top_p, int32_t *out_tokens, int32_t *out_num_accepted,
                                        void *workspace, size_t workspace_bytes, void *stream, float *row_sum,
                                        float *p_draft)
{
    return run(target_logits, logits_dtype, T, V, logits_row_stride, draft_probs, q_row_stride, draft_ids,
               cu_num_draft, B, uniforms, temperature, out_tokens, out_num_accepted, workspace, workspace_bytes,
               static_cast<cudaStream_t>(stream), nullptr, row_sum, nullptr, p_draft, nullptr, nullptr, 0, top_k,
               top_p);
}

spec_status spec_reject_sample_ex(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                  int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                  const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                  const float *uniforms, const float *temperature, int32_t *out_tokens,
                                  int32_t *out_num_accepted, void *workspace, size_t workspace_bytes, void *stream,
                                  const spec_reject_options *options)
{
    const spec_reject_options none = {};
    const spec_reject_options &o = options ? *options : none;
    return run(target_logits, logits_dtype, T, V, logits_row_stride, draft_probs, q_row_stride, draft_ids,
               cu_num_draft, B, uniforms, temperature, out_tokens, out_num_accepted, workspace, workspace_bytes,
               static_cast<cudaStream_t>(stream), nullptr, o.row_sum, nullptr, o.p_draft, nullptr, nullptr, 0,
               o.top_k, o.top_p, o.counters);
}

spec_status spec_reject_debug_rowstats(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                       int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                       const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                       const float *uniforms, const float *temperature, int32_t *out_tokens,
                                       int32_t *out_num_accepted, void *workspace, size_t workspace_bytes,
                                       void *stream, float *row_max, float *row_sum, int32_t *row_argmax,
                                       float *p_draft, float *z_out)
{
    return run(target_logits, logits_dtype, T, V, logits_row_stride, draft_probs, q_row_stride, draft_ids,
               cu_num_draft, B, uniforms, temperature, out_tokens, out_num_accepted, workspace, workspace_bytes,
               static_cast<cudaStream_t>(stream), row_max, row_sum, row_argmax, p_draft, z_out);
}

spec_status spec_reject_sample_profiled(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                        int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                        const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                        const float *uniforms, const float *temperature, int32_t *out_tokens,
                                        int32_t *out_num_accepted, void *workspace, size_t workspace_bytes,
                                        void *stream, const int32_t *top_k, const float *top_p,
                                        void *const *stage_events, int num_events)
{
    return run(target_logits, logits_dtype, T, V, logits_row_stride, draft_probs, q_row_stride, draft_ids,
               cu_num_draft, B, uniforms, temperature, out_tokens, out_num_accepted, workspace, workspace_bytes,
               static_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr, nullptr, nullptr,
               reinterpret_cast<cudaEvent_t *>(const_cast<void **>(stage_events)), num_events, top_k, top_p);
}

spec_status spec_reject_last_device_error(const void *workspace, void *stream, int32_t *error_bits,
                                          int32_t *first_bad_request)
{
    if (!workspace)
        return SPEC_ERR_INVALID_ARG;
    const char *base =
        reinterpret_cast<const char *>((reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255));
    int32_t word[2] = {0, INT_MAX};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(word, base, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SPEC_ERR_CUDA;
    if (error_bits)
        *error_bits = word[0];
    if (first_bad_request)
        *first_bad_request = (word[0] & SPEC_DEVERR_LAYOUT) || word[1] == INT_MAX ? -1 : word[1];
    return word[0] ? SPEC_ERR_DEVICE_INPUT : SPEC_OK;
}

size_t spec_reject_host_arena_size(int32_t B, int64_t T, int32_t V, spec_dtype logits_dtype, int has_draft_probs)
{
    Plan pl;
    if (!make_plan(B, T, V, logits_dtype, has_draft_probs, &pl))
        return 0;
    const size_t es = logits_dtype == SPEC_BF16 ? 2 : 4;
    size_t o = 0;
    o = align256(o + es * (size_t)T * (size_t)V);                                       // logits
    o = align256(o + (has_draft_probs ? 4 * (size_t)(T - B) * (size_t)V : 0));          // draft probs
    o = align256(o + 4 * (size_t)(T - B));                                              // draft ids
    o = align256(o + 4 * (size_t)(B + 1));                                              // cu
    o = align256(o + 8 * (size_t)T);                                                    // uniforms
    o = align256(o + 4 * (size_t)B);                                                    // temperature
    o = align256(o + 4 * (size_t)T);                                                    // out tokens
    o = align256(o + 4 * (size_t)B);                                                    // out accepted
    o = align256(o + 8 * (size_t)B + 8 * (size_t)SPEC_METRIC_COUNT);                    // top-k, top-p, counters
    return o + pl.total + 256;
}

spec_status spec_reject_sample_host(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                    const float *draft_probs, const int32_t *draft_ids, const int32_t *cu_num_draft,
                                    int32_t B, const float *uniforms, const float *temperature, int32_t *out_tokens,
                                    int32_t *out_num_accepted, void *device_arena, size_t arena_bytes, void *stream)
{
    return spec_reject_sample_host_ex(target_logits, logits_dtype, T, V, draft_probs, draft_ids, cu_num_draft, B,
                                      uniforms, temperature, out_tokens, out_num_accepted, device_arena, arena_bytes,
                                      stream, nullptr, nullptr, nullptr);
}

spec_status spec_reject_sample_host_ex(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                       const float *draft_probs, const int32_t *draft_ids,
                                       const int32_t *cu_num_draft, int32_t B, const float *uniforms,
                                       const float *temperature, int32_t *out_tokens, int32_t *out_num_accepted,
                                       void *device_arena, size_t arena_bytes, void *stream, const int32_t *top_k,
                                       const float *top_p, int64_t *counters)
{
    if (!device_arena || !cu_num_draft || B < 0 || T < B || V < 1 || (T > 0 && (!target_logits || !uniforms ||
        !out_tokens)) || (B > 0 && (!temperature || !out_num_accepted)) || (T > B && !draft_ids))
        return SPEC_ERR_INVALID_ARG;
    const size_t need = spec_reject_host_arena_size(B, T, V, logits_dtype, draft_probs != nullptr);
    if (need == 0)
        return SPEC_ERR_INVALID_ARG;
    if (arena_bytes < need)
        return SPEC_ERR_WORKSPACE;
    if (cuda_error_pending())  // before the pointer queries below, which clear their own errors
        return SPEC_ERR_CUDA;
    const size_t es = logits_dtype == SPEC_BF16 ? 2 : 4;
    const int has_q = draft_probs != nullptr;
    char *a = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(device_arena) + 255) & ~uintptr_t(255));
    size_t o = 0;
    char *d_logits = a + o;
    o = align256(o + es * (size_t)T * (size_t)V);
    float *d_q = reinterpret_cast<float *>(a + o);
    o = align256(o + (has_q ? 4 * (size_t)(T - B) * (size_t)V : 0));
    int32_t *d_ids = reinterpret_cast<int32_t *>(a + o);
    o = align256(o + 4 * (size_t)(T - B));
    int32_t *d_cu = reinterpret_cast<int32_t *>(a + o);
    o = align256(o + 4 * (size_t)(B + 1));
    float *d_uni = reinterpret_cast<float *>(a + o);
    o = align256(o + 8 * (size_t)T);
    float *d_temp = reinterpret_cast<float *>(a + o);
    o = align256(o + 4 * (size_t)B);
    int32_t *d_tok = reinterpret_cast<int32_t *>(a + o);
    o = align256(o + 4 * (size_t)T);
    int32_t *d_acc = reinterpret_cast<int32_t *>(a + o);
    o = align256(o + 4 * (size_t)B);
    int32_t *d_topk = reinterpret_cast<int32_t *>(a + o);
    float *d_topp = reinterpret_cast<float *>(a + o + 4 * (size_t)B);
    int64_t *d_ctr = reinterpret_cast<int64_t *>(a + o + 8 * (size_t)B);  // 8-byte aligned
    o = align256(o + 8 * (size_t)B + 8 * (size_t)SPEC_METRIC_COUNT);
    char *d_ws = a + o;
    const size_t ws_bytes = arena_bytes - (size_t)(d_ws - reinterpret_cast<char *>(device_arena));

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Draft probabilities in pinned, mapped host memory are read in place over the host link:
    // the kernels touch only q(x*) of each verify row and the row at each request's first
    // rejection, a small part of the [T - B, V] array.  Pageable memory is copied whole.
    auto mapped = [](const void *p) -> const void * {  // device address of pinned, mapped host memory
        cudaPointerAttributes pa{};
        if (cudaPointerGetAttributes(&pa, p) == cudaSuccess && pa.type == cudaMemoryTypeHost && pa.devicePointer)
            return pa.devicePointer;
        (void)cudaGetLastError();
        return nullptr;
    };
    const float *q_in_place = has_q ? static_cast<const float *>(mapped(draft_probs)) : nullptr;
    // Pinned logits too, and a batch that takes the first-rejection pass: that pass reads the
    // target rows in place as well, only the rows up to each request's output row.
    const void *logits_in_place = (T > 0) ? mapped(target_logits) : nullptr;
    const bool filtered = top_k || top_p;
    const bool all_in_place = logits_in_place && (!has_q || q_in_place) && B >= SPEC_KL_MIN_REQUESTS &&
                              aligned(logits_in_place, 16) && ((size_t)V * es) % 16 == 0 &&
                              (!filtered || logits_dtype == SPEC_BF16);
    // one cudaMemcpyAsync per buffer
    const struct {
        void *dst;
        const void *src;
        size_t bytes;
    } in[] = {
        {d_logits, target_logits, all_in_place ? 0 : es * (size_t)T * (size_t)V},
        {d_q, draft_probs, has_q && !q_in_place ? 4 * (size_t)(T - B) * (size_t)V : 0},
        {d_ids, draft_ids, 4 * (size_t)(T - B)},
        {d_cu, cu_num_draft, 4 * (size_t)(B + 1)},
        {d_uni, uniforms, 8 * (size_t)T},
        {d_temp, temperature, 4 * (size_t)B},
        {d_topk, top_k, top_k ? 4 * (size_t)B : 0},
        {d_topp, top_p, top_p ? 4 * (size_t)B : 0},
        {d_ctr, counters, counters ? 8 * (size_t)SPEC_METRIC_COUNT : 0},
    };
    for (const auto &c : in)
        if (c.bytes && cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return SPEC_ERR_CUDA;
    // q in place: K2 reads q(x*) over the link, then the rows K3 needs are staged into the
    // arena's q region (the rest of it stays unwritten)
    spec_status st =
        all_in_place
            ? run(logits_in_place, logits_dtype, T, V, V, q_in_place, V, d_ids, d_cu, B, d_uni, d_temp, d_tok, d_acc,
                  d_ws, ws_bytes, s, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0, top_k ? d_topk : nullptr,
                  top_p ? d_topp : nullptr, counters ? d_ctr : nullptr, has_q ? d_q : nullptr, true, d_logits)
            : run(d_logits, logits_dtype, T, V, V, has_q ? (q_in_place ? q_in_place : d_q) : nullptr, V, d_ids, d_cu,
                  B, d_uni, d_temp, d_tok, d_acc, d_ws, ws_bytes, s, nullptr, nullptr, nullptr, nullptr, nullptr,
                  nullptr, 0, top_k ? d_topk : nullptr, top_p ? d_topp : nullptr, counters ? d_ctr : nullptr,
                  q_in_place ? d_q : nullptr);
    if (st != SPEC_OK)
        return st;
    if ((T && cudaMemcpyAsync(out_tokens, d_tok, 4 * (size_t)T, cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
        (B && cudaMemcpyAsync(out_num_accepted, d_acc, 4 * (size_t)B, cudaMemcpyDeviceToHost, s) != cudaSuccess) ||
        (counters && cudaMemcpyAsync(counters, d_ctr, 8 * (size_t)SPEC_METRIC_COUNT, cudaMemcpyDeviceToHost, s) !=
                         cudaSuccess) ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

// ---------------------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory
// ---------------------------------------------------------------------------------------

// Scratch for spec_reject_sample_noalloc(): a fixed device array instead of a caller
// workspace.  Every GPU that loads this library holds it until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_REJECT_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on each device.  In host code the symbol is only a
// host-side stand-in, so the address comes from cudaGetSymbolAddress, looked up once per device
// (std::call_once: concurrent first calls from several host threads are safe).  The address
// belongs to the device's primary context as the library's module was loaded into it: after
// cudaDeviceReset() on a device the module is loaded again and this entry must not be called
// on that device any more in this process (the cached address would be stale).
static void *g_noalloc_addr[kMaxDevices];
static std::once_flag g_noalloc_once[kMaxDevices];

spec_status spec_reject_sample_noalloc(const void *target_logits, spec_dtype logits_dtype, int64_t T, int32_t V,
                                       int64_t logits_row_stride, const float *draft_probs, int64_t q_row_stride,
                                       const int32_t *draft_ids, const int32_t *cu_num_draft, int32_t B,
                                       const float *uniforms, const float *temperature, int32_t *out_tokens,
                                       int32_t *out_num_accepted, int32_t *device_error_word, void *stream)
{
    // the same argument checks as spec_reject_sample(), first, so that both entries return the
    // same status for the same bad argument (the scratch stands in for the workspace pointer)
    spec_status st = check_args(target_logits, logits_dtype, T, V, logits_row_stride, draft_probs, q_row_stride,
                                draft_ids, cu_num_draft, B, uniforms, temperature, out_tokens, out_num_accepted,
                                g_noalloc_scratch);
    if (st != SPEC_OK)
        return st;
    const size_t need = spec_reject_workspace_size(B, T, V, logits_dtype, draft_probs != nullptr);
    if (need == 0)
        return SPEC_ERR_INVALID_ARG;
    if (need > SPEC_REJECT_NOALLOC_SCRATCH_BYTES)
        return SPEC_ERR_WORKSPACE;  // batch too large for the fixed scratch array
    int dev;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return SPEC_ERR_CUDA;
    if (cuda_error_pending())
        return SPEC_ERR_CUDA;
    std::call_once(g_noalloc_once[dev], [dev]() {  // with `dev` current
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) == cudaSuccess)
            g_noalloc_addr[dev] = addr;
    });
    if (!g_noalloc_addr[dev])
        return SPEC_ERR_CUDA;
    // Nothing in the scratch has to start at zero: the first kernel of every call writes the
    // error word and clears every counter and queue the later kernels use, and every other
    // region is written before it is read.
    st = spec_reject_sample(target_logits, logits_dtype, T, V, logits_row_stride, draft_probs, q_row_stride,
                            draft_ids, cu_num_draft, B, uniforms, temperature, out_tokens, out_num_accepted,
                            g_noalloc_addr[dev], SPEC_REJECT_NOALLOC_SCRATCH_BYTES, stream);
    if (st != SPEC_OK || !device_error_word)
        return st;
    // the error word sits at the start of the (256-byte aligned) scratch
    if (cudaMemcpyAsync(device_error_word, g_noalloc_addr[dev], 2 * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SPEC_ERR_CUDA;
    return SPEC_OK;
}

spec_status spec_reject_metrics_update(const int32_t *cu_num_draft, const int32_t *out_num_accepted, int32_t B,
                                       int64_t *counters, void *stream)
{
    if (B < 0 || !counters || (B > 0 && (!cu_num_draft || !out_num_accepted)) || !aligned(counters, 8) ||
        !aligned(cu_num_draft, 4) || !aligned(out_num_accepted, 4))
        return SPEC_ERR_INVALID_ARG;
    if (B == 0)
        return SPEC_OK;
    DeviceInfo *di;
    if (cuda_error_pending() || device_info(&di) != cudaSuccess)
        return SPEC_ERR_CUDA;
    const int grid = (int)clamp_grid(di->sms, (B + kThreads - 1) / kThreads);
    metrics_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        cu_num_draft, out_num_accepted, B, reinterpret_cast<unsigned long long *>(counters));
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_ngram_propose(const int32_t *tokens, const int64_t *cu_tokens, int32_t B, int32_t min_n,
                               int32_t max_n, int32_t k, int64_t max_model_len, int32_t *out_drafts,
                               int32_t *out_num_drafts, void *stream)
{
    if (B < 0 || min_n < 1 || max_n < min_n || max_n > SPEC_NGRAM_MAX_N || k < 1 || k > SPEC_REJECT_MAX_SPEC_LEN)
        return SPEC_ERR_INVALID_ARG;
    if (B == 0)
        return SPEC_OK;
    if (!tokens || !cu_tokens || !out_drafts || !out_num_drafts || !aligned(tokens, 4) || !aligned(cu_tokens, 8) ||
        !aligned(out_drafts, 4) || !aligned(out_num_drafts, 4))
        return SPEC_ERR_INVALID_ARG;
    DeviceInfo *di;
    if (cuda_error_pending() || device_info(&di) != cudaSuccess)
        return SPEC_ERR_CUDA;
    const int grid = (int)clamp_grid((int64_t)di->sms * 8, B);
    ngram_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(tokens, cu_tokens, B, min_n, max_n, k,
                                                                            max_model_len, out_drafts, out_num_drafts);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Tree workspace: the sampler's plan for N one-row "requests" (error word, partials), then
// an all-zero cu_num_draft [N + 1] and temperature [N] that make K1 take the argmax of
// every node row.
static bool tree_plan(int64_t N, int32_t B, int32_t V, spec_dtype dt, Plan *pl, size_t *off_cu, size_t *off_temp,
                      size_t *total)
{
    if (N < 0 || N > INT32_MAX - 1 || B < 0 || !make_plan((int32_t)N, N, V, dt, 0, pl))
        return false;
    *off_cu = align256(pl->total);
    *off_temp = align256(*off_cu + sizeof(int32_t) * (size_t)(N + 1));
    *total = align256(*off_temp + sizeof(float) * (size_t)(N > 0 ? N : 1)) + 256;
    return true;
}

size_t spec_tree_workspace_size(int64_t N, int32_t B, int32_t V, spec_dtype logits_dtype)
{
    Plan pl;
    size_t oc, ot, total;
    return tree_plan(N, B, V, logits_dtype, &pl, &oc, &ot, &total) ? total : 0;
}

spec_status spec_tree_verify_greedy(const void *target_logits, spec_dtype logits_dtype, int64_t N, int32_t V,
                                    int64_t logits_row_stride, const int32_t *parent, const int32_t *node_tokens,
                                    const int32_t *cu_nodes, int32_t B, int32_t *out_tokens,
                                    int32_t *out_num_accepted, int32_t *out_last_node, void *workspace,
                                    size_t workspace_bytes, void *stream)
{
    Plan pl;
    size_t off_cu, off_temp, total;
    if ((logits_dtype != SPEC_F32 && logits_dtype != SPEC_BF16) || V < 1 || V > SPEC_REJECT_MAX_VOCAB ||
        !tree_plan(N, B, V, logits_dtype, &pl, &off_cu, &off_temp, &total))
        return SPEC_ERR_INVALID_ARG;
    if (!workspace || !cu_nodes || (N > 0 && (!target_logits || !parent || !node_tokens || !out_tokens)) ||
        (B > 0 && (!out_num_accepted || !out_last_node)) || (logits_row_stride != 0 && logits_row_stride < V))
        return SPEC_ERR_INVALID_ARG;
    const size_t es = logits_dtype == SPEC_BF16 ? 2 : 4;
    if (!aligned(target_logits, es) || !aligned(parent, 4) || !aligned(node_tokens, 4) || !aligned(cu_nodes, 4) ||
        !aligned(out_tokens, 4) || !aligned(out_num_accepted, 4) || !aligned(out_last_node, 4))
        return SPEC_ERR_INVALID_ARG;
    if (workspace_bytes < total)
        return SPEC_ERR_WORKSPACE;
    DeviceInfo *di;
    if (cuda_error_pending() || device_info(&di) != cudaSuccess)
        return SPEC_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *base = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255));
    int32_t *fcu = reinterpret_cast<int32_t *>(base + off_cu);
    float *ftemp = reinterpret_cast<float *>(base + off_temp);
    if (cudaMemsetAsync(fcu, 0, (off_temp - off_cu) + sizeof(float) * (size_t)(N > 0 ? N : 1), st) != cudaSuccess)
        return SPEC_ERR_CUDA;
    Params P{};
    P.logits = target_logits;
    P.T = N;
    P.V = V;
    P.lstride = logits_row_stride;
    P.cu = fcu;
    P.B = (int32_t)N;
    P.temp = ftemp;
    P.part = reinterpret_cast<float2 *>(base + pl.off_part);
    P.err = reinterpret_cast<int32_t *>(base + pl.off_err);
    P.chunk = pl.chunk;
    P.nchunks = pl.nchunks;
    const int DT = logits_dtype == SPEC_BF16 ? 1 : 0;
    const int64_t full = (int64_t)di->sms * (di->blocks_rowstats[DT] > 0 ? di->blocks_rowstats[DT] : 1);
    const int gridA = (int)clamp_grid(full, (N * (int64_t)pl.nchunks + kWarps - 1) / kWarps);
    launch_rowstats(DT, P, *di, N, pl.nchunks, target_logits, logits_row_stride, gridA, st, 1);
    if (B > 0)
        tree_walk_kernel<<<(B + kWarps - 1) / kWarps, kThreads, 0, st>>>(P, parent, node_tokens, cu_nodes, B,
                                                                        out_tokens, out_num_accepted, out_last_node);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

const char *spec_reject_status_string(spec_status status)
{
    switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument (null pointer, size, stride or alignment)";
    case SPEC_ERR_UNSUPPORTED: return "unsupported size";
    case SPEC_ERR_WORKSPACE: return "workspace too small";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_DEVICE_INPUT: return "invalid device input (see the device error word)";
    case SPEC_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int spec_reject_version(void) { return 100; }

int spec_reject_blocks_per_request(spec_dtype logits_dtype, int32_t B, int32_t V)
{
    Plan pl;
    DeviceInfo *di;
    if (B < 1 || !make_plan(B, B, V, logits_dtype, 0, &pl) || device_info(&di) != cudaSuccess)
        return 0;
    return 1 << lazy_cluster_log2(*di, logits_dtype == SPEC_BF16 ? 1 : 0, B, pl.nchunks);
}

int spec_reject_launches_per_call(spec_dtype logits_dtype, int32_t B, int32_t V, int has_draft_probs,
                                  int has_filters)
{
    Plan pl;
    DeviceInfo *di;
    const int stages = spec_reject_num_kernels(logits_dtype, B, has_draft_probs, has_filters);
    if (B < 1 || !make_plan(B, B, V, logits_dtype, has_draft_probs, &pl) || device_info(&di) != cudaSuccess)
        return stages;
    const int DT = logits_dtype == SPEC_BF16 ? 1 : 0;
    if (has_filters) {  // with cuts: bf16 rows of at least SPEC_KL_MIN_REQUESTS requests take the pass
        const int64_t n16 = lazy_cut16_requests(*di, B);
        return stages == 2 && n16 > 0 && n16 < B ? 3 : stages;
    }
    if (lazy_cluster_log2(*di, DT, B, pl.nchunks) == 0 && lazy_tail_requests(*di, DT, B, pl.nchunks) > 0)
        return 3;  // the layout check, the first-rejection pass, its chained second launch
    return stages;
}

int spec_reject_num_kernels(spec_dtype logits_dtype, int32_t B, int has_draft_probs, int has_filters)
{
    if (B >= (has_filters ? SPEC_KL_MIN_REQUESTS : 1) && (!has_filters || logits_dtype == SPEC_BF16))
        return 2;  // layout check, then the pass up to each first rejection
    return (has_filters ? 3 : 2) + (has_draft_probs ? 1 : 0);
}

}  // extern "C"

#endif  // SPEC_KL_CUT_VARIANT
