// queue.cu -- KW, the work-queue first-rejection pass of the rejection sampler (sm_103a).
//
// What it computes is the sampler of include/spec_reject.h ("第12章 投机解码：以小博大"
// §12.2.1-§12.2.4, §12.3.2): per request, accept draft x*_i while u * q_i(x*) < p_i(x*),
// stop at the first rejection j ("vllm v1 源码精读（五）" §7), draw the recovered token from
// max(0, p_j - q_j) (one-hot q: p_j without x*, §12.9) or the bonus token from p_k.  Only
// the target rows up to each request's output row are needed, since the test at position i
// reads row t_i alone and the scan stops at j.
//
// How: every warp of the grid works through a queue of items, independently of the others.
//   row item       up to kQRowGroup chunks (8 KB of logits each) of one target row, streamed
//                  through the warp's ring of TMA bulk-copy slots and reduced to the same
//                  per-chunk partials as K1 (softmax (m_c, s_c) or greedy (max, argmax)).
//   residual item  up to kQResGroup units of kQResTokens tokens of a rejected output row: the
//                  target logits and the draft probabilities of the unit land in one slot (two
//                  bulk copies) and reduce to sum max(0, p - q) over the unit.
// A per-row counter gathers the chunks of a row; the warp whose chunk completes the row (and
// whose row is the request's next undecided one: the decision of row i - 1 adds one to row
// i's counter when it accepts) decides position i with K2's arithmetic.  An acceptance
// publishes the row wq_depth positions further on (rows are streamed that far ahead of the
// decisions: depth 1 streams only rows that are certainly needed); a rejection or the bonus
// row draws the output token in the same warp (K2's chunk scan and warp descent), except an
// explicit-q recovery, which publishes the residual items of its row and is drawn by the warp
// that completes the last of them.  Rows of the first wq_depth positions of every request are
// listed by the set-up kernel (the "fresh" rows); everything later is published into the
// queue while the pass runs.  A warp that needs work takes a published item first, so that a
// request's next row and its residual pass (whose target row is then still in L2) run soon
// after the decision that made them, and fresh rows otherwise.
//
// Synchronisation: a warp never waits for another warp while it holds work that someone
// waits for.  A warp with nothing to do polls the queue with a bounded wait (it gives up
// after a fixed time and sets SPEC_DEVERR_TIMEOUT) until an item is published or every
// request is finished.  Every mbarrier wait is bounded too.

#include <cuda_runtime.h>
#include <stdint.h>
#include <limits.h>
#include <math.h>

#include "spec_reject.h"
#include "common.cuh"

namespace specrej {
namespace {

#ifndef SPEC_WQ_WORKERS
#define SPEC_WQ_WORKERS 4     // worker warps per block, each with its own ring (plus one scheduler warp)
#endif
#ifndef SPEC_WQ_STAGES
#define SPEC_WQ_STAGES 3      // ring slots per warp
#endif
#ifndef SPEC_WQ_MIN_BLOCKS
#define SPEC_WQ_MIN_BLOCKS 2  // blocks per SM: 2 x 4 warps x 3 slots x 8 KB = 192 KB in flight per SM
#endif
#ifndef SPEC_WQ_POLL_NS
#define SPEC_WQ_POLL_NS 2000000000ull  // a warp waiting for work gives up after this long
#endif
constexpr int kQWorkers = SPEC_WQ_WORKERS;
constexpr int kQStages = SPEC_WQ_STAGES;
constexpr int kQThreads = (kQWorkers + 1) * 32;
constexpr size_t kQSmem = (size_t)kQWorkers * kQStages * kUnitBytes;
constexpr int kQResQOffset = kUnitBytes / 2;  // byte offset of a residual unit's draft probabilities
static_assert(kQResTokens * 4 <= kUnitBytes / 2, "a residual unit's target logits and draft probabilities share a slot");

// Control words
constexpr int kCtlFresh = 0;   // fresh row items claimed
constexpr int kCtlHead = 2;    // queue entries claimed (head and tail are read together)
constexpr int kCtlTail = 3;    // queue entries reserved by publishers
constexpr int kCtlDone = 4;    // requests finished (outputs written, or reported invalid)
constexpr int kCtlNFresh = 5;  // fresh row items listed by the set-up kernel

constexpr int kKindRow = 0, kKindRes = 1;

// An item of work: 16 bytes, each half with its top bit set so that a reader can tell a
// written entry from a cleared one (the queue is cleared by the set-up kernel of every call).
//   a: 1 | kind (3) | position i (6) | k_r saturated at 63 (6) | item index g (16) | temperature bits (32)
//   b: 1 | request r (31) | target row t (32)
struct Item {
    int kind, i, k, g, r;
    uint32_t t;
    float temp;
};

__device__ __forceinline__ ulonglong2 encode(const Item &it)
{
    ulonglong2 e;
    e.x = (1ull << 63) | ((unsigned long long)it.kind << 60) | ((unsigned long long)it.i << 54) |
          ((unsigned long long)min(it.k, 63) << 48) | ((unsigned long long)it.g << 32) |
          (unsigned long long)__float_as_uint(it.temp);
    e.y = (1ull << 63) | ((unsigned long long)(uint32_t)it.r << 32) | (unsigned long long)it.t;
    return e;
}

__device__ __forceinline__ Item decode(ulonglong2 e)
{
    Item it;
    it.kind = (int)((e.x >> 60) & 7);
    it.i = (int)((e.x >> 54) & 63);
    it.k = (int)((e.x >> 48) & 63);
    it.g = (int)((e.x >> 32) & 0xffff);
    it.temp = __uint_as_float((uint32_t)e.x);
    it.r = (int)((e.y >> 32) & 0x7fffffff);
    it.t = (uint32_t)e.y;
    return it;
}

__device__ __forceinline__ bool written(ulonglong2 e) { return (e.x >> 63) && (e.y >> 63); }

__device__ __forceinline__ ulonglong2 ld_volatile16(const ulonglong2 *p)
{
    ulonglong2 v;
    asm volatile("ld.volatile.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_volatile16(ulonglong2 *p, ulonglong2 v)
{
    asm volatile("st.volatile.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(v.x), "l"(v.y) : "memory");
}

__device__ __forceinline__ uint2 ld_volatile_u2(const uint32_t *p)
{
    uint2 v;
    asm volatile("ld.volatile.global.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_volatile_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.volatile.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: the pass may start while the set-up kernel finishes; it waits
// here for the set-up kernel's writes before it reads any of them.
__device__ __forceinline__ void wait_for_prerequisite() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Chunk masses of a row relative to 2^M from the partials other warps wrote in this launch
// (read past L1), one chunk optionally replaced.
struct PartialsL2 {
    const float2 *pp;
    float cs, M;
    int override_chunk;
    float override_mass;
    __device__ __forceinline__ float operator()(int c) const
    {
        if (c == override_chunk)
            return override_mass;
        const float2 pc = __ldcg(pp + c);
        return (pc.x == -INFINITY) ? 0.f : pc.y * ex2(pc.x * cs - M);
    }
};

// ---------------------------------------------------------------------------------------
// Set-up kernel: clear the counters and the queue, check the layout, list the fresh rows
// ---------------------------------------------------------------------------------------

// Exclusive prefix sum over the 256 threads of a block (and the block total).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t &total)
{
    __shared__ uint32_t s_w[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        s_w[warp] = incl;
    __syncthreads();
    uint32_t before = 0, all = 0;
    for (int w = 0; w < 8; ++w) {
        const uint32_t x = s_w[w];
        before += w < warp ? x : 0;
        all += x;
    }
    __syncthreads();  // s_w is reused by the next call
    total = all;
    return before + incl - v;
}

__global__ void __launch_bounds__(256) wq_init_kernel(Params P)
{
    allow_dependents();  // the pass may be scheduled now; it waits for this grid's writes
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nth = (int64_t)gridDim.x * blockDim.x;
    for (int64_t x = tid; x < P.T; x += nth)
        P.wq_cnt[x] = 0;
    if (P.rcnt)
        for (int64_t x = tid; x < P.B; x += nth)
            P.rcnt[x] = 0;
    for (int64_t x = tid; x < (int64_t)P.wq_cap; x += nth)
        P.wq_dq[x] = make_ulonglong2(0ull, 0ull);
    if (blockIdx.x != 0)
        return;

    validate_layout(P);  // error word: [0] bits, [1] first bad request
    __syncthreads();
    const bool layout_bad = (P.err[0] & SPEC_DEVERR_LAYOUT) != 0;
    uint32_t nrows = 0;
    if (layout_bad) {  // the whole batch is invalid: nothing is streamed
        for (int r = threadIdx.x; r < P.B; r += blockDim.x)
            P.out_acc[r] = -1;
    } else {
        // fresh rows, level by level (position 0 of every request first): position i of
        // request r is listed when i < min(depth, k_r + 1); a request with k_r > 32 lists its
        // row 0 only (its decision reports the error)
        const int per = (P.B + (int)blockDim.x - 1) / (int)blockDim.x;
        const int r0 = min(P.B, (int)threadIdx.x * per), r1 = min(P.B, r0 + per);
        for (int lvl = 0; lvl < P.wq_depth; ++lvl) {
            uint32_t mine = 0;
            for (int r = r0; r < r1; ++r) {
                const int k = P.cu[r + 1] - P.cu[r];
                const int n = k > SPEC_REJECT_MAX_SPEC_LEN ? 1 : min(P.wq_depth, k + 1);
                mine += lvl < n;
            }
            uint32_t total;
            uint32_t pos = nrows + block_excl_scan(mine, total);
            for (int r = r0; r < r1; ++r) {
                const int k = P.cu[r + 1] - P.cu[r];
                const int n = k > SPEC_REJECT_MAX_SPEC_LEN ? 1 : min(P.wq_depth, k + 1);
                if (lvl == 0)
                    P.rstate[r] = n - 1;  // last position listed (published) for the request
                if (lvl < n) {
                    Item it;
                    it.kind = kKindRow;
                    it.i = lvl;
                    it.k = k;
                    it.g = 0;
                    it.r = r;
                    it.t = (uint32_t)(P.cu[r] + r + lvl);
                    it.temp = P.temp[r];
                    P.wq_fresh[pos++] = encode(it);
                }
            }
            nrows += total;
            if (total == 0)
                break;
        }
    }
    if (threadIdx.x == 0) {
        P.wq_ctl[kCtlFresh] = 0;
        P.wq_ctl[kCtlHead] = 0;
        P.wq_ctl[kCtlTail] = 0;
        P.wq_ctl[kCtlDone] = layout_bad ? (uint32_t)P.B : 0u;
        P.wq_ctl[kCtlNFresh] = nrows * (uint32_t)P.wq_row_items;
    }
}

// ---------------------------------------------------------------------------------------
// The pass
// ---------------------------------------------------------------------------------------
//
// A block is one scheduler warp and kQWorkers worker warps.  The scheduler claims items from
// the global queue and the fresh rows, in batches and off the workers' critical path, and
// keeps a small block-local queue in shared memory filled (about one item per worker); a
// worker pops its next item from there while its ring still holds the current item's units.

constexpr int kQHi = 2 * kQWorkers;  // block-local entries from the global queue (served first)
constexpr int kQLo = 4 * kQWorkers;  // block-local entries of fresh rows

// What a ring slot holds (written by lane 0 before its copies are issued; the mbarrier's
// release / acquire makes it visible to the lanes that wait on the slot).
struct SlotMeta {
    int32_t t, r, unit;   // target row, request, chunk (row item) or residual unit
    int16_t kind, i, k, last;
    float temp;
    int32_t nunits;       // units of the item (counted at its last unit)
};

// A block-local ring of items: the scheduler writes entries, then advances `tail`; a worker
// reads the entry at `head` and claims it by advancing `head` (compare-and-swap).
template <int N> struct LocalRing {
    ulonglong2 e[N];
    unsigned head, tail;
};

struct BlockQueue {
    LocalRing<kQHi> hi;
    LocalRing<kQLo> lo;
    int exit;     // set by the scheduler once every request is finished
    int spec_ok;  // set by the scheduler while the fresh rows are used up and the queue runs low
};

__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ int atom_add_acq_rel(int32_t *p, int v)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned ld_volatile_smem(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}

__device__ __forceinline__ void st_volatile_smem(unsigned *p, unsigned v)
{
    asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

__device__ __forceinline__ ulonglong2 ld_volatile_smem16(const ulonglong2 *p)
{
    ulonglong2 v;
    asm volatile("ld.volatile.shared.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "r"(smem_addr(p)) : "memory");
    return v;
}

__device__ __forceinline__ ulonglong2 with_index(ulonglong2 e, uint32_t g)
{
    e.x = (e.x & ~(0xffffull << 32)) | ((unsigned long long)g << 32);
    return e;
}

// Appends the entries of the lanes with `have` set to ring R (warp; the caller made sure they
// fit).  Returns how many.
template <int N> __device__ __forceinline__ int ring_push(LocalRing<N> &R, unsigned tail, bool have, ulonglong2 e,
                                                          int lane)
{
    const unsigned b = __ballot_sync(kFull, have);
    if (have)
        R.e[(tail + __popc(b & ((1u << lane) - 1u))) % N] = e;
    __syncwarp();
    __threadfence_block();
    if (lane == 0 && b)
        st_volatile_smem(&R.tail, tail + __popc(b));
    return __popc(b);
}

// Takes one entry of ring R (one thread); false when it is empty.
template <int N> __device__ __forceinline__ bool ring_pop(LocalRing<N> &R, ulonglong2 &e)
{
    for (int a = 0; a < 4; ++a) {
        const unsigned h = ld_volatile_smem(&R.head);
        if (h == ld_volatile_smem(&R.tail))
            return false;
        __threadfence_block();
        e = ld_volatile_smem16(&R.e[h % N]);
        if (atomicCAS(&R.head, h, h + 1) == h)
            return true;
    }
    return false;
}

// Scheduler warp: keeps the block-local rings filled until every request is finished.  Items
// the global queue has published go to the `hi` ring (about one per worker, so that a
// request's next row or residual pass starts soon), fresh rows to the `lo` ring in batches.
__device__ __noinline__ void schedule(const Params &P, BlockQueue &Q, int lane)
{
    uint32_t *ctl = P.wq_ctl;
    const uint32_t nfresh = __ldcg(ctl + kCtlNFresh);
    bool fresh_done = false;
    int64_t pend = -1;  // per lane: a claimed queue entry not yet written
    uint64_t idle_since = global_ns();
    unsigned backoff = 32;
    for (;;) {
        bool progress = false;
        unsigned hit = ld_volatile_smem(&Q.hi.tail);
        const int hi_queued = (int)(hit - ld_volatile_smem(&Q.hi.head));
        int hi_free = kQHi - hi_queued;
        int hi_want = kQWorkers - hi_queued;
        // (a) claimed entries that have been written since
        ulonglong2 e = make_ulonglong2(0ull, 0ull);
        bool ready = false;
        if (pend >= 0) {
            e = ld_volatile16(P.wq_dq + pend);
            ready = written(e);
        }
        const unsigned rb = __ballot_sync(kFull, ready);
        if (rb && hi_free > 0) {
            const bool take = ready && __popc(rb & ((1u << lane) - 1u)) < hi_free;
            if (take) {
                fence_acq_rel();  // acquire: what the publisher wrote before the entry
                pend = -1;
            }
            const int n = ring_push(Q.hi, hit, take, e, lane);
            hit += n;
            hi_free -= n;
            hi_want -= n;
            progress = true;
        }
        // (b) claim entries the global queue has published, one per lane
        const unsigned anypend = __ballot_sync(kFull, pend >= 0);
        uint2 ht = make_uint2(0, 0);
        if (lane == 0)
            ht = ld_volatile_u2(ctl + kCtlHead);
        ht.x = __shfl_sync(kFull, ht.x, 0);
        ht.y = __shfl_sync(kFull, ht.y, 0);
        const uint32_t backlog = ht.y - min(ht.x, ht.y);
        if (hi_want > 0 && !anypend && backlog > 0) {
            const int m = min(min(hi_want, 32), (int)backlog);
            uint32_t h0 = 0;
            if (lane == 0)
                h0 = atomicAdd(ctl + kCtlHead, (uint32_t)m);
            h0 = __shfl_sync(kFull, h0, 0);
            if (lane < m && h0 + lane < P.wq_cap)
                pend = (int64_t)h0 + lane;
            continue;  // poll them at once
        }
        // (c) fresh rows, in batches, while the `lo` ring is at most half full
        if (!fresh_done) {
            const unsigned lot = ld_volatile_smem(&Q.lo.tail);
            const int lo_queued = (int)(lot - ld_volatile_smem(&Q.lo.head));
            if (lo_queued <= kQLo / 2) {
                const int m = min(kQLo - lo_queued, 32);
                uint32_t f0 = 0;
                if (lane == 0)
                    f0 = atomicAdd(ctl + kCtlFresh, (uint32_t)m);
                f0 = __shfl_sync(kFull, f0, 0);
                const uint32_t f = f0 + lane;
                const bool ok = lane < m && f < nfresh;
                if (ok) {
                    const uint32_t row = f / (uint32_t)P.wq_row_items;
                    e = with_index(__ldg(P.wq_fresh + row), f - row * (uint32_t)P.wq_row_items);
                }
                progress = ring_push(Q.lo, lot, ok, e, lane) > 0 || progress;
                if (f0 + (uint32_t)m >= nfresh)
                    fresh_done = true;
            }
        }
        // deeper read-ahead while the fresh rows are used up and little is queued
        if (lane == 0)
            st_volatile_smem(reinterpret_cast<unsigned *>(&Q.spec_ok),
                             fresh_done && backlog < (uint32_t)P.wq_spare_items ? 1u : 0u);
        if (progress) {
            backoff = 32;
            idle_since = global_ns();
            continue;
        }
        if (ld_volatile_u32(ctl + kCtlDone) >= (uint32_t)P.B)
            break;
        if (global_ns() - idle_since > SPEC_WQ_POLL_NS) {
            if (lane == 0)
                atomicOr(P.err, SPEC_DEVERR_TIMEOUT);
            break;
        }
        __nanosleep(backoff);
        backoff = min(backoff * 2, 256u);
    }
    __syncwarp();
    if (lane == 0)
        st_volatile_smem(reinterpret_cast<unsigned *>(&Q.exit), 1u);
}

// Publishes items for request r (warp): `nrows` row entries for positions i0, i0 + 1, ...
// (kKindRow, wq_row_items items each), or the residual items of its output row t
// (kKindRes).  Writes the warp made before (residual statistics, the published-row mark)
// are ordered before the entries.
__device__ __forceinline__ void publish(const Params &P, int lane, int kind, uint32_t t, int r, int i0, int nrows,
                                       int k, float temp)
{
    const int per = kind == kKindRow ? P.wq_row_items : P.wq_res_items;
    const int n = kind == kKindRow ? nrows * per : per;
    __syncwarp();
    fence_acq_rel();
    uint32_t base = 0;
    if (lane == 0)
        base = atomicAdd(P.wq_ctl + kCtlTail, (uint32_t)n);
    base = __shfl_sync(kFull, base, 0);
    Item it;
    it.kind = kind;
    it.k = k;
    it.r = r;
    it.temp = temp;
    for (int x = lane; x < n; x += 32) {
        const int dr = kind == kKindRow ? x / per : 0;
        it.i = i0 + dr;
        it.t = t + (uint32_t)dr;
        it.g = x - dr * per;
        if (base + (uint32_t)x < P.wq_cap)
            st_volatile16(P.wq_dq + base + x, encode(it));
    }
}

// Writes request r's outputs (warp): accepted drafts, the token at j, -1 after; the counters.
__device__ __forceinline__ void write_outputs(const Params &P, int lane, int r, int64_t tb, int64_t db, int k, int j,
                                              int token)
{
    const int xs = lane < j ? __ldg(P.ids + db + lane) : -1;
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
    if (lane == 0)
        atomicAdd(P.wq_ctl + kCtlDone, 1u);
}

// A request reported invalid (k_r > 32, or a draft id outside [0, V)): -1 outputs.
__device__ __forceinline__ void write_invalid(const Params &P, int lane, int r, int64_t tb, int k, int bits)
{
    for (int64_t i = lane; i <= k; i += 32)
        P.out_tokens[tb + i] = -1;
    if (lane == 0) {
        P.out_acc[r] = -1;
        atomicOr(P.err, bits);
        atomicMin(P.err + 1, r);
        atomicAdd(P.wq_ctl + kCtlDone, 1u);
    }
}

// Masses held in registers, lane l holding entries l, l + 32, ...: the warp's total and the
// inverse-CDF locate, with the arithmetic (and so the results) of chunk_total / chunk_locate.
constexpr int kRegMasses = 8;  // entries per lane: up to 256 chunks or residual units
__device__ __forceinline__ float regs_total(const float (&m)[kRegMasses], int n, int lane)
{
    float carry = 0.f;
#pragma unroll
    for (int j = 0; j < kRegMasses; ++j)
        if (32 * j < n) {
            const float incl = warp_incl_scan(32 * j + lane < n ? m[j] : 0.f, lane);
            carry += __shfl_sync(kFull, incl, 31);
        }
    return carry;
}

__device__ __forceinline__ int regs_locate(const float (&m)[kRegMasses], int n, float theta, int lane, float &theta_in)
{
    float carry = 0.f;
    int last_pos = -1;
#pragma unroll
    for (int j = 0; j < kRegMasses; ++j)
        if (32 * j < n) {
            const float mj = 32 * j + lane < n ? m[j] : 0.f;
            const float incl = warp_incl_scan(mj, lane) + carry;
            const unsigned hit = __ballot_sync(kFull, incl > theta);
            if (hit) {
                const int L = __ffs(hit) - 1;
                theta_in = theta - __shfl_sync(kFull, incl - mj, L);
                return 32 * j + L;
            }
            const unsigned pos = __ballot_sync(kFull, mj > 0.f);
            if (pos)
                last_pos = 32 * j + 31 - __clz(pos);
            carry = __shfl_sync(kFull, incl, 31);
        }
    theta_in = INFINITY;
    return last_pos < 0 ? n - 1 : last_pos;
}

// The decision at row t = t_i of request r (warp), and, while the next row is already
// reduced, the decisions after it.  Ends with the request's outputs, with its residual items
// published, or with the next row still streaming.
template <int DT>
__device__ __noinline__ void decide(const Params &P, BlockQueue &Q, uint32_t t, int r, int i, int k, float temp,
                                    int lane)
{
    const bool greedy = !(temp > 0.f);
    const float cs = greedy ? 0.f : kLog2e / temp;
    const int64_t tb = (int64_t)t - i;  // the request's first target row
    const int64_t db = tb - r;          // its first draft row
    const int NC = P.nchunks;
    const bool in_regs = NC <= 32 * kRegMasses;
    if (i == 0) {  // per-request checks, as K2
        int kk = k;
        const bool bad_len = k > SPEC_REJECT_MAX_SPEC_LEN;
        if (bad_len)
            kk = P.cu[r + 1] - P.cu[r];  // the item carries k saturated at 63
        const int xs = (!bad_len && lane < k) ? __ldg(P.ids + db + lane) : 0;
        const unsigned badid = __ballot_sync(kFull, !bad_len && lane < k && (xs < 0 || xs >= P.V));
        if (bad_len || badid) {
            write_invalid(P, lane, r, tb, kk, bad_len ? SPEC_DEVERR_SPEC_LEN : SPEC_DEVERR_DRAFT_ID);
            return;
        }
    }
    for (;;) {
        const float2 *pp = P.part + (int64_t)t * NC;
        const char *row = row_ptr<DT>(P, t);
        // inputs of the test at position i (lane 0), issued before the partials are combined;
        // lane 1: the last position published for the request
        int xs = -1, published = 0;
        float ua = 0.f, ls = 0.f, qs = 1.f;
        if (lane == 1 && i < k)
            published = __ldcg(P.rstate + r);
        if (lane == 0 && i < k) {
            xs = __ldg(P.ids + db + i);
            if (!greedy) {
                ua = __ldg(P.uni + 2 * (int64_t)t);
                ls = load1<DT>(row, xs);
                if (P.q)
                    qs = __ldg(P.q + (db + i) * P.qstride + xs);
            }
        }
        float2 pc[kRegMasses];
        if (in_regs) {
#pragma unroll
            for (int j = 0; j < kRegMasses; ++j)
                if (32 * j + lane < NC)
                    pc[j] = __ldcg(pp + 32 * j + lane);
        }
        // the row's statistics (K2's per-row combine)
        float m = -INFINITY, sv = 0.f, best = -INFINITY;
        int idx = INT_MAX;
        auto add = [&](float2 c2) {
            if (greedy) {
                const int cix = __float_as_int(c2.y);
                if (c2.x > best || (c2.x == best && cix < idx)) {
                    best = c2.x;
                    idx = cix;
                }
            } else if (c2.x != -INFINITY) {
                const float Mc = c2.x * cs;
                if (Mc > m) {
                    sv = (m == -INFINITY) ? c2.y : sv * ex2(m - Mc) + c2.y;
                    m = Mc;
                } else {
                    sv += c2.y * ex2(Mc - m);
                }
            }
        };
        if (in_regs) {
#pragma unroll
            for (int j = 0; j < kRegMasses; ++j)
                if (32 * j + lane < NC)
                    add(pc[j]);
        } else {
            for (int c = lane; c < NC; c += 32)
                add(__ldcg(pp + c));
        }
        int am = 0;
        float Mi = 0.f, Si = 0.f;
        bool accept;
        if (greedy) {
            warp_argmax(best, idx);
            am = idx == INT_MAX ? 0 : idx;
            accept = i < k && __shfl_sync(kFull, xs, 0) == am;
        } else {
            const float mw = warp_max(m);
            const float sw = warp_sum(m == -INFINITY ? 0.f : sv * ex2(m - mw));
            Mi = mw;
            Si = sw;
            accept = false;
            if (lane == 0 && i < k) {
                const float e = fmaf(ls, cs, -Mi);
                const float wstar = ex2(e);
                const double lhs = (double)ua * (double)qs;  // exact
                const float ps = wstar / Si;
                if (ps > 1e-30f || wstar == 0.f)
                    accept = lhs < (double)ps;
                else  // below fp32's normal range: form p(x*) in double
                    accept = lhs < exp2((double)e) / (double)Si;
            }
            accept = __shfl_sync(kFull, accept, 0);
        }
        if (accept) {
            // rows streamed ahead of the decisions: wq_depth, deeper while the fresh rows are used
            // up and the global queue runs low (the GPU would idle otherwise; the scheduler
            // keeps that flag)
            const int depth =
                ld_volatile_smem(reinterpret_cast<const unsigned *>(&Q.spec_ok)) ? max(P.wq_depth, P.wq_tail_depth)
                                                                                 : P.wq_depth;
            const int upto = min(k, i + depth);
            const int done_upto = __shfl_sync(kFull, published, 1);
            if (upto > done_upto) {
                if (lane == 0)
                    P.rstate[r] = upto;
                publish(P, lane, kKindRow, (uint32_t)(tb + done_upto + 1), r, done_upto + 1, upto - done_upto, k,
                        temp);
            }
            // position i + 1 may be decided once its row is reduced: count this decision in
            int go = 0;
            if (lane == 0)
                go = atom_add_acq_rel(P.wq_cnt + t + 1, 1) + 1 == NC + 1;
            if (!__shfl_sync(kFull, go, 0))
                return;  // the warp that reduces its last chunk decides it
            fence_acq_rel();
            ++t;
            ++i;
            continue;
        }

        // ---- the output token at row t_j, j = i
        const int j = i;
        int token = -1;
        if (greedy) {
            token = am;
        } else if (j < k && P.q) {  // explicit q: the residual pass, drawn by its last warp
            if (lane == 0)
                P.rstat[r] = make_float2(Mi, Si);
            publish(P, lane, kKindRes, t, r, j, 1, k, temp);
            return;
        } else {
            const float us = __ldg(P.uni + 2 * (int64_t)t + 1);
            int64_t excl = -1;
            int cx = -1;
            float mx = 0.f;
            if (j < k) {  // one-hot draft: the residual is p without x*
                const int xj = __shfl_sync(kFull, xs, 0);
                cx = xj / P.chunk;
                TargetMass<DT, false> fx{row, cs, Mi, xj, 0u};
                mx = warp_range_mass(fx, (int64_t)cx * P.chunk, min((int64_t)P.V, (int64_t)(cx + 1) * P.chunk), lane);
                excl = xj;
            }
            float th;
            int c;
            if (in_regs) {
                float ms[kRegMasses];
#pragma unroll
                for (int jj = 0; jj < kRegMasses; ++jj) {
                    const int cc = 32 * jj + lane;
                    ms[jj] = cc == cx ? mx : ((cc >= NC || pc[jj].x == -INFINITY) ? 0.f : pc[jj].y * ex2(pc[jj].x * cs - Mi));
                }
                float Z = regs_total(ms, NC, lane);
                if (!(Z > 0.f) && cx >= 0) {  // empty residual: draw from p itself
#pragma unroll
                    for (int jj = 0; jj < kRegMasses; ++jj) {
                        const int cc = 32 * jj + lane;
                        if (cc == cx)
                            ms[jj] = (pc[jj].x == -INFINITY) ? 0.f : pc[jj].y * ex2(pc[jj].x * cs - Mi);
                    }
                    Z = regs_total(ms, NC, lane);
                    excl = -1;
                }
                c = regs_locate(ms, NC, us * Z, lane, th);
            } else {
                PartialsL2 cm{pp, cs, Mi, cx, mx};
                float Z = chunk_total(cm, NC, lane);
                if (!(Z > 0.f) && cx >= 0) {
                    cm.override_chunk = -1;
                    Z = chunk_total(cm, NC, lane);
                    excl = -1;
                }
                c = chunk_locate(cm, NC, us * Z, lane, th);
            }
            TargetMass<DT, false> f{row, cs, Mi, excl, 0u};
            token = (int)warp_find(f, (int64_t)c * P.chunk, min((int64_t)P.V, (int64_t)(c + 1) * P.chunk), th, lane);
        }
        write_outputs(P, lane, r, tb, db, k, j, token);
        return;
    }
}

// The explicit-q recovery of request r at its output row t = t_j, once every residual unit
// of the row is reduced (warp).
template <int DT>
__device__ __noinline__ void draw_residual(const Params &P, uint32_t t, int r, int j, int k, float temp, int lane)
{
    const float cs = kLog2e / temp;
    const int64_t tb = (int64_t)t - j, db = tb - r;
    const float2 st = __ldcg(P.rstat + r);
    const float Mj = st.x, Sj = st.y;
    const float us = __ldg(P.uni + 2 * (int64_t)t + 1);
    const char *rowj = row_ptr<DT>(P, t);
    const float *rp = P.rpart + (int64_t)r * P.wq_nres;
    const int NU = P.wq_nres;
    float Z, th = 0.f;
    int u = 0;
    if (NU <= 32 * kRegMasses) {
        float ms[kRegMasses];
#pragma unroll
        for (int jj = 0; jj < kRegMasses; ++jj)
            ms[jj] = 32 * jj + lane < NU ? __ldcg(rp + 32 * jj + lane) : 0.f;
        Z = regs_total(ms, NU, lane);
        if (Z > 0.f)
            u = regs_locate(ms, NU, us * Z, lane, th);
    } else {
        const ChunkMassFromL2 cmz{rp};
        Z = chunk_total(cmz, NU, lane);
        if (Z > 0.f)
            u = chunk_locate(cmz, NU, us * Z, lane, th);
    }
    int token;
    if (Z > 0.f) {
        const ResidualMass<DT, false> f{rowj, P.q + (db + j) * P.qstride, cs, Mj, 1.f / Sj, 0u};
        token = (int)warp_find(f, (int64_t)u * kQResTokens, min((int64_t)P.V, (int64_t)(u + 1) * kQResTokens), th,
                               lane);
    } else {  // empty residual: draw from p itself
        const PartialsL2 cm{P.part + (int64_t)t * P.nchunks, cs, Mj, -1, 0.f};
        const float Zp = chunk_total(cm, P.nchunks, lane);
        const int c = chunk_locate(cm, P.nchunks, us * Zp, lane, th);
        const TargetMass<DT, false> f{rowj, cs, Mj, -1, 0u};
        token = (int)warp_find(f, (int64_t)c * P.chunk, min((int64_t)P.V, (int64_t)(c + 1) * P.chunk), th, lane);
    }
    write_outputs(P, lane, r, tb, db, k, j, token);
}

// Residual mass of one unit that has landed in a slot: target logits at byte 0, draft
// probabilities at kQResQOffset; tokens the bulk copies left out (a ragged end) come from
// global memory.
template <int DT>
__device__ __forceinline__ float residual_unit(const unsigned char *slot, const char *row, const float *qrow,
                                               int64_t v0, int nt, float cs, float M, float inv_s, int lane)
{
    constexpr int ES = Elem<DT>::kSize;
    const ResidualMass<DT, false> f{row, qrow, cs, M, inv_s, 0u};
    const int cov_t = (int)(((uint32_t)nt * ES) & ~15u) / ES;
    const int cov_q = (int)(((uint32_t)nt * 4) & ~15u) / 4;
    const int groups = min(cov_t, cov_q) / 4;  // 4-token groups read from the slot
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int g = lane; g < groups; g += 32) {
        float x[4];
        if (DT == 1) {
            const uint2 w = *reinterpret_cast<const uint2 *>(slot + (size_t)g * 8);
            x[0] = __uint_as_float(w.x << 16);
            x[1] = __uint_as_float(w.x & 0xffff0000u);
            x[2] = __uint_as_float(w.y << 16);
            x[3] = __uint_as_float(w.y & 0xffff0000u);
        } else {
            const float4 w = *reinterpret_cast<const float4 *>(slot + (size_t)g * 16);
            x[0] = w.x;
            x[1] = w.y;
            x[2] = w.z;
            x[3] = w.w;
        }
        const float4 q4 = *reinterpret_cast<const float4 *>(slot + kQResQOffset + (size_t)g * 16);
        acc[0] += fmaxf(0.f, f.pm(x[0]) - q4.x);
        acc[1] += fmaxf(0.f, f.pm(x[1]) - q4.y);
        acc[2] += fmaxf(0.f, f.pm(x[2]) - q4.z);
        acc[3] += fmaxf(0.f, f.pm(x[3]) - q4.w);
    }
    for (int v = groups * 4 + lane; v < nt; v += 32)
        acc[0] += f.one(v0 + v);
    return warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
}

// Worker warp: streams its items' units through its ring, reduces them, and decides / draws
// when a unit completes a row or a residual pass.
template <int DT>
__device__ __forceinline__ void work(const Params &P, BlockQueue &Q, unsigned char *slots, uint64_t *bars,
                                     SlotMeta *meta, int lane)
{
    constexpr int ES = Elem<DT>::kSize;
    constexpr int VEC = Elem<DT>::kVec;
    const int NC = P.nchunks;

    // ---- issue side (lane 0): the current item, its units still to issue, the next item
    Item cur{}, nxt{};
    int iu = 0, ie = 0;
    bool have_nxt = false;
    uint32_t qi = 0;  // units issued

    auto pop = [&](Item &it) -> bool {
        if (ld_volatile_smem(reinterpret_cast<const unsigned *>(&Q.exit)))
            return false;  // every request is finished: what is left in the rings is not needed
        ulonglong2 e;
        if (ring_pop(Q.hi, e) || ring_pop(Q.lo, e)) {
            it = decode(e);
            return true;
        }
        return false;
    };
    auto issue_unit = [&](const Item &it, int u, bool last, int nunits) {
        const int s = (int)(qi % kQStages);
        SlotMeta &mt = meta[s];
        mt.t = (int32_t)it.t;
        mt.r = it.r;
        mt.unit = u;
        mt.kind = (int16_t)it.kind;
        mt.i = (int16_t)it.i;
        mt.k = (int16_t)it.k;
        mt.last = (int16_t)last;
        mt.temp = it.temp;
        mt.nunits = nunits;
        unsigned char *dst = slots + (size_t)s * kUnitBytes;
        const char *row = row_ptr<DT>(P, it.t);
        if (it.kind == kKindRow) {
            const int64_t lo = (int64_t)u * P.chunk;
            const int64_t hi = min((int64_t)P.V, lo + P.chunk);
            const uint32_t bytes = (uint32_t)((hi - lo) * ES) & ~15u;
            mbar_arrive_expect_tx(&bars[s], bytes);
            if (bytes)
                bulk_g2s(dst, row + lo * ES, bytes, &bars[s]);
        } else {
            const int64_t lo = (int64_t)u * kQResTokens;
            const int64_t nt = min((int64_t)P.V - lo, (int64_t)kQResTokens);
            const uint32_t bt = (uint32_t)(nt * ES) & ~15u;
            const uint32_t bq = (uint32_t)(nt * 4) & ~15u;
            const float *qrow = P.q + ((int64_t)it.t - it.r) * P.qstride;  // draft row d = t - r
            mbar_arrive_expect_tx(&bars[s], bt + bq);
            if (bt)
                bulk_g2s(dst, row + lo * ES, bt, &bars[s]);
            if (bq)
                bulk_g2s(dst + kQResQOffset, qrow + lo, bq, &bars[s]);
        }
        ++qi;
    };
    // lane 0: issue until the ring is full or no item is at hand; take the next item from the
    // block's queue while the ring is full
    auto fill = [&](uint32_t qc) {
        while (qi - qc < (uint32_t)kQStages) {
            if (iu == ie) {
                if (!have_nxt && !pop(nxt))
                    return;
                cur = nxt;
                have_nxt = false;
                iu = cur.g * (cur.kind == kKindRow ? kQRowGroup : kQResGroup);
                ie = min(cur.kind == kKindRow ? NC : P.wq_nres,
                         iu + (cur.kind == kKindRow ? kQRowGroup : kQResGroup));
            }
            const int lo = cur.g * (cur.kind == kKindRow ? kQRowGroup : kQResGroup);
            issue_unit(cur, iu, iu + 1 == ie, ie - lo);
            ++iu;
        }
        if (!have_nxt && iu == ie)
            have_nxt = pop(nxt);
    };

    // ---- completion of the latest finished item, acted on one unit later
    bool have_pend = false;
    int pend_old = 0;  // lane 0: the counter before this item's units were added
    SlotMeta pend_meta{};
    auto settle = [&]() {
        if (!have_pend)
            return;
        have_pend = false;
        const SlotMeta &pm = pend_meta;
        const int thr = pm.kind == kKindRow ? NC + (pm.i > 0 ? 1 : 0) : P.wq_nres;
        if (!__shfl_sync(kFull, pend_old + pm.nunits == thr, 0))
            return;
        fence_acq_rel();
        if (pm.kind == kKindRow)
            decide<DT>(P, Q, (uint32_t)pm.t, pm.r, pm.i, pm.k, pm.temp, lane);
        else
            draw_residual<DT>(P, (uint32_t)pm.t, pm.r, pm.i, pm.k, pm.temp, lane);
    };

    // ---- consume side (whole warp)
    uint32_t qc = 0;
    float last_temp = NAN, cs = 0.f;
    bool greedy = true;
    int res_r = -1;  // request whose residual statistics are cached
    float res_M = 0.f, res_inv_s = 0.f;
    bool ok = true;
    for (;;) {
        if (lane == 0)
            fill(qc);
        if (__shfl_sync(kFull, qi, 0) == qc) {
            settle();  // its decision may publish the work this warp is about to wait for
            // nothing in flight: wait for the scheduler's next item, or for the end
            int st = 0;
            if (lane == 0) {
                const uint64_t t0 = global_ns();
                for (;;) {
                    if (pop(nxt)) {
                        have_nxt = true;
                        st = 1;
                        break;
                    }
                    if (ld_volatile_smem(reinterpret_cast<const unsigned *>(&Q.exit))) {
                        st = 0;
                        break;
                    }
                    if (global_ns() - t0 > SPEC_WQ_POLL_NS) {
                        atomicOr(P.err, SPEC_DEVERR_TIMEOUT);
                        st = -1;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            if (__shfl_sync(kFull, st, 0) <= 0)
                break;
            continue;
        }
        const int s = (int)(qc % kQStages);
        if (!__all_sync(kFull, mbar_wait(&bars[s], (qc / kQStages) & 1, P.err))) {
            ok = false;
            break;
        }
        const SlotMeta mt = meta[s];
        const unsigned char *slot = slots + (size_t)s * kUnitBytes;
        if (have_pend && !mt.last) {
            // act on the previous item's count now, with this unit landed but not yet read: the
            // slot stays untouched until this unit is reduced below
            settle();
        }
        const char *row = row_ptr<DT>(P, (uint32_t)mt.t);
        if (mt.temp != last_temp) {
            last_temp = mt.temp;
            greedy = !(mt.temp > 0.f);
            cs = greedy ? 0.f : kLog2e / mt.temp;
        }
        if (mt.kind == kKindRow) {
            const int c = mt.unit;
            UnitRange R;
            R.lo = (int64_t)c * P.chunk;
            R.hi = min((int64_t)P.V, R.lo + P.chunk);
            R.vlo = R.lo;
            R.nvec = ((R.hi - R.lo) * ES) / 16;
            R.vhi = R.vlo + R.nvec * VEC;
            const uint4 *stage = reinterpret_cast<const uint4 *>(slot);
            uint4 v[kVecPerLane];
#pragma unroll
            for (int kk = 0; kk < kVecPerLane; ++kk) {
                const int vi = kk * 32 + lane;
                v[kk] = (vi < R.nvec) ? stage[vi] : neg_inf_vec<DT>();
            }
            __syncwarp();
            ++qc;
            if (lane == 0)
                fill(qc);  // the slot is in registers: refill it
            float2 *out = P.part + (int64_t)mt.t * NC + c;
            if (greedy)
                argmax_regs<DT>(out, lane, v, R, row);
            else
                softmax_regs<DT>(out, cs, lane, v, R, row);
        } else {
            if (mt.r != res_r) {
                const float2 st = __ldcg(P.rstat + mt.r);
                res_r = mt.r;
                res_M = st.x;
                res_inv_s = 1.f / st.y;
            }
            const int64_t v0 = (int64_t)mt.unit * kQResTokens;
            const int nt = (int)min((int64_t)P.V - v0, (int64_t)kQResTokens);
            const float *qrow = P.q + ((int64_t)mt.t - mt.r) * P.qstride;
            const float z = residual_unit<DT>(slot, row, qrow, v0, nt, cs, res_M, res_inv_s, lane);
            __syncwarp();
            ++qc;
            if (lane == 0) {
                P.rpart[(int64_t)mt.r * P.wq_nres + mt.unit] = z;
                fill(qc);
            }
        }
        if (mt.last) {
            // the item is done: count it in now, act on the count after the next unit (the
            // atomic's round trip overlaps that unit)
            settle();
            if (lane == 0) {
                if (mt.kind == kKindRow)
                    pend_old = atom_add_acq_rel(P.wq_cnt + mt.t, mt.nunits);
                else
                    pend_old = atom_add_acq_rel(P.rcnt + mt.r, mt.nunits);
            }
            pend_meta = mt;
            have_pend = true;
        }
    }
    settle();
    // gave up on a wait: let this warp's copies still in flight land before exiting
    if (!ok && lane == 0)
        for (uint32_t q2 = qc + 1; q2 < qi; ++q2)
            mbar_wait(&bars[q2 % kQStages], (q2 / kQStages) & 1, P.err);
}

template <int DT>
__global__ void __launch_bounds__(kQThreads, SPEC_WQ_MIN_BLOCKS) wq_kernel(Params P)
{
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kQWorkers * kQStages];
    __shared__ SlotMeta smeta[kQWorkers * kQStages];
    __shared__ BlockQueue Q;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x < kQWorkers * kQStages)
        mbar_init(&full[threadIdx.x], 1);
    if (threadIdx.x == 0) {
        Q.hi.head = Q.hi.tail = 0;
        Q.lo.head = Q.lo.tail = 0;
        Q.exit = 0;
        Q.spec_ok = 0;
    }
    mbar_fence_init();
    __syncthreads();  // the only block-wide barrier: from here on the warps are independent
    wait_for_prerequisite();
    if (warp == 0) {
        schedule(P, Q, lane);
    } else {
        const int w = warp - 1;
        work<DT>(P, Q, ring + (size_t)w * kQStages * kUnitBytes, full + w * kQStages, smeta + w * kQStages, lane);
    }
}

}  // namespace

cudaError_t queue_pass_occupancy(int DT, int *blocks_per_sm)
{
    cudaError_t e;
    if (DT) {
        if ((e = cudaFuncSetAttribute(wq_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQSmem)))
            return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, wq_kernel<1>, kQThreads, kQSmem);
    }
    if ((e = cudaFuncSetAttribute(wq_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kQSmem)))
        return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, wq_kernel<0>, kQThreads, kQSmem);
}

cudaError_t launch_queue_pass(const Params &P, int DT, int sms, int blocks_per_sm, cudaStream_t stream,
                              cudaEvent_t between)
{
    // set-up: enough blocks to clear the queue quickly
    const int64_t words = (int64_t)P.wq_cap + P.T;
    const int init_grid = (int)max((int64_t)1, min((int64_t)sms * 4, (words + 2047) / 2048));
    wq_init_kernel<<<init_grid, 256, 0, stream>>>(P);
    cudaError_t e = cudaGetLastError();
    if (e)
        return e;
    if (between && (e = cudaEventRecord(between, stream)))
        return e;
    const int64_t max_blocks = kQMaxWarps / (kQWorkers + 1);
    const int grid = (int)max((int64_t)1, min((int64_t)sms * blocks_per_sm, max_blocks));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kQThreads, 1, 1);
    cfg.dynamicSmemBytes = kQSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = between ? 0 : 1;
    return DT ? cudaLaunchKernelEx(&cfg, wq_kernel<1>, P) : cudaLaunchKernelEx(&cfg, wq_kernel<0>, P);
}

}  // namespace specrej
