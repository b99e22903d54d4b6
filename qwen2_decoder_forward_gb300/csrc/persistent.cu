// Persistent single-launch decode step for one sequence (batch 1).
//
// One CTA per SM, all resident (cooperative launch).  Each CTA owns a fixed
// slice of every weight matrix: the Q/K/V, o_proj and gate/up row pairs and
// the down_proj and LM-head rows, split evenly over the CTAs.  The CTA's
// slices stream, in the order they are used, through a ring of six 28 KB
// shared-memory stages filled by bulk (TMA) copies with mbarriers, issued by
// one lane of a feeding warpgroup, so the weight stream runs ahead of the
// compute and never waits for activations; each compute warp waits for a
// stage when it reads it and releases it when its dot products are done.
// The feeding warpgroup hands its registers to the two compute warpgroups
// (setmaxnreg), which then need not spill.  The compute warps run the
// steps of the layer (minfer "Qwen2 / Qwen2.5 Architecture Support",
// section 1) and exchange activation vectors through global "packets":
// 64-bit words holding a float and the launch's epoch, written and read
// with single-copy atomic 64-bit accesses, so a reader that sees the
// current epoch has the value.  A per-phase arrival counter, polled by one
// thread per CTA, tells a consumer when to read the larger exchanges.
//
// Per layer the dependencies are x -> Q/K/V (norm needs all of x), q/k/v ->
// attention units (kv head, key chunk, query heads), the units' partials
// -> the merge of head h by CTA h -> o, broadcast to every CTA -> o_proj,
// x -> gate/up (norm), SiLU(gate)*up -> down.  The arithmetic is the
// per-step kernels' own (rowdot.cuh, attn.cuh), so the logits are
// bit-identical to the multi-kernel path.
//
// Every wait is bounded (2 s of the global timer): a wait that gives up
// raises kGuardTimeout, and the CTA stops, waits for its copies in flight
// and returns.
#include "attn.cuh"
#include "ctx.h"
#include "persistent.h"
#include "rowdot.cuh"
#include "sm100.cuh"

namespace qwen2 {

namespace {

constexpr int kCompute = 256;            // warpgroups 0-1: the compute warps
constexpr int kThreads = 384;            // + warpgroup 2, whose first lane feeds the weight ring
// Register split (setmaxnreg): launched at 168 per thread (384 x 168 =
// 64512); the feeding warpgroup drops to 40 and the compute warpgroups rise
// to 232: 4 x 32 x 40 + 8 x 32 x 232 = 64512, the launch's own total.
constexpr int kRegFeed = 40, kRegCompute = 232;
typedef unsigned long long u64;

// Every bounded wait of a launch gives up after wait_limit() ns: 2 s
// (kPersistWaitNs) unless the test hook shortened it for one launch.
__shared__ u64 wait_limit_s;
__device__ __forceinline__ u64 wait_limit() { return wait_limit_s; }

// The asynchronous-proxy primitives of sm100.cuh (mbarriers, bulk copies)
// and its global timer.
using sm100::bulk_g2s;
using sm100::mbar_arrive;
using sm100::mbar_expect_tx;
using sm100::mbar_init;
using sm100::mbar_test;
using sm100::mbar_try_wait;
__device__ __forceinline__ u64 now_ns() { return sm100::global_ns(); }

// Named-barrier OR over the 256 compute threads.
__device__ __forceinline__ bool compute_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void pk_put(u64* p, float v, unsigned ep) {
    const u64 w = ((u64)ep << 32) | (u64)__float_as_uint(v);
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ u64 pk_raw(const u64* p) {
    u64 w;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
    return w;
}

// Per-phase arrival counters: every CTA adds 1 when it has written its
// packets of a phase; a consumer CTA has one thread wait until the counter
// reaches epoch * CTAs and then reads the packets once (each packet still
// carries its epoch, so an early counter only costs a re-poll).  Polling
// one line with one thread per CTA is far cheaper than every thread
// polling the packets themselves.
constexpr int kCntStride = 16;  // one 128-byte line per counter
__device__ __forceinline__ void cnt_arrive(u64* cnt) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], 1;" ::"l"(cnt) : "memory");
}

// Reader of packets of one epoch; after a failed wait it returns 0 at once
// and the thread's `failed` flag stays set.
struct PkReader {
    unsigned ep;
    bool failed = false;
    __device__ __forceinline__ float get(const u64* p) {
        if (failed) return 0.f;
        u64 w = pk_raw(p);
        if ((unsigned)(w >> 32) == ep) return __uint_as_float((unsigned)w);
        const u64 t0 = now_ns();
        while ((unsigned)(w >> 32) != ep) {
            if (now_ns() - t0 > wait_limit()) {
                failed = true;
                return 0.f;
            }
            __nanosleep(32);
            w = pk_raw(p);
        }
        return __uint_as_float((unsigned)w);
    }
};

// Read n packets with all of a thread's loads in flight at once (element j
// at addr(j) goes to store(j, value)).  Packets not yet of this epoch are
// all polled again together, so a thread waits about one L2 round trip
// after the last of its packets lands.  Threads of the 256-thread compute
// group take elements tid, tid + 256, ...
template <int KMAX, class Addr, class Store, class Idle>
__device__ __forceinline__ void pk_gather(PkReader& rd, int n, Addr addr, Store store, Idle idle) {
    const int tid = threadIdx.x;
    for (int j0 = 0; j0 < n; j0 += KMAX * 256) {
        u64 w[KMAX];
        unsigned pending = 0;
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int j = j0 + tid + 256 * k;
            if (j < n) w[k] = pk_raw(addr(j));
        }
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            const int j = j0 + tid + 256 * k;
            if (j < n) {
                if ((unsigned)(w[k] >> 32) == rd.ep) store(j, __uint_as_float((unsigned)w[k]));
                else pending |= 1u << k;
            }
        }
        if (pending && !rd.failed) {
            const u64 t0 = now_ns();
            while (pending) {
                idle();
                __nanosleep(100);
#pragma unroll
                for (int k = 0; k < KMAX; ++k)
                    if (pending & (1u << k)) w[k] = pk_raw(addr(j0 + tid + 256 * k));
#pragma unroll
                for (int k = 0; k < KMAX; ++k)
                    if ((pending & (1u << k)) && (unsigned)(w[k] >> 32) == rd.ep) {
                        store(j0 + tid + 256 * k, __uint_as_float((unsigned)w[k]));
                        pending &= ~(1u << k);
                    }
                if (pending && now_ns() - t0 > wait_limit()) {
                    rd.failed = true;
                    break;
                }
            }
        }
        if (rd.failed) {
#pragma unroll
            for (int k = 0; k < KMAX; ++k)
                if (pending & (1u << k)) store(j0 + tid + 256 * k, 0.f);
        }
    }
}

__device__ __forceinline__ int split(int n, int c, int G) { return (int)(((long long)n * c) / G); }


}  // namespace

// Packet buffer layout per layer (offsets in packets).  Every buffer is
// written kPkRep times; CTA c reads copy c % kPkRep, so the reads of the
// 152 CTAs spread over kPkRep times more L2 lines.
constexpr int kPkRep = 4;
struct PkLayout {
    int qkv, x1, m, x2, att, per_layer;          // offsets of copy 0
    int n_qkv, n_x, n_m, n_att, n_o;             // packets per copy
    __host__ __device__ PkLayout(int nqkv, int H, int I, int nh, int max_chunks) {
        n_qkv = nqkv;
        n_x = H;
        n_m = I;
        n_att = nh * max_chunks * kPartStride;
        n_o = nh * kHd;
        qkv = 0;
        x1 = qkv + kPkRep * n_qkv;
        m = x1 + kPkRep * n_x;
        x2 = m + kPkRep * n_m;
        att = x2 + kPkRep * n_x;
        per_layer = att + kPkRep * n_att;
    }
    // The merged attention output of layer l (long context), kept after
    // all layers' buffers and the argmax pairs of `grid` CTAs: placing it
    // inside each layer's block shifted the hot buffers and cost about 5 %
    // at short context (measured).
    __host__ __device__ size_t o_base(int L, int grid, int l) const {
        return (size_t)L * per_layer + 2 * (size_t)grid + (size_t)l * kPkRep * n_o;
    }
};

// The weight stream of one CTA: its slices of every matrix, in the order the
// compute uses them, cut into chunks of rows_h (K = H) or rows_i (K = I)
// rows, one chunk per ring stage.  Thread 0 calls refill() whenever it is
// about to wait; refill never blocks: it issues bulk copies into every stage
// the compute has released, in order.
struct Feeder {
    const PersistentArgs* a;
    unsigned char* ring;
    uint64_t* full;
    uint64_t* empty;
    int c, G;
    int l = 0, ph = 0, r = 0, r1 = 0;  // next chunk: layer (L: LM head), phase, row range
    int issued = 0;
    bool done = false;

    __device__ __forceinline__ void range() {
        const int H = a->H, I = a->I;
        if (l == a->L) {
            r = split(a->V, c, G);
            r1 = split(a->V, c + 1, G);
        } else if (ph == 0) {
            r = 2 * split(a->nqkv / 2, c, G);
            r1 = 2 * split(a->nqkv / 2, c + 1, G);
        } else if (ph == 1) {
            r = 2 * split(H / 2, c, G);
            r1 = 2 * split(H / 2, c + 1, G);
        } else if (ph == 2) {
            r = 2 * split(I, c, G);
            r1 = 2 * split(I, c + 1, G);
        } else {
            r = split(H, c, G);
            r1 = split(H, c + 1, G);
        }
    }
    __device__ __forceinline__ void init(const PersistentArgs* a_, unsigned char* ring_, uint64_t* full_, uint64_t* empty_,
                                         int c_, int G_) {
        a = a_;
        ring = ring_;
        full = full_;
        empty = empty_;
        c = c_;
        G = G_;
        range();
    }
    __device__ __forceinline__ void refill() {
        while (!done) {
            while (r >= r1) {  // next phase with rows
                if (l == a->L) {
                    done = true;
                    return;
                }
                if (++ph == 4) {
                    ph = 0;
                    ++l;
                }
                range();
            }
            const int s = issued % a->stages;
            const unsigned k = issued / a->stages;
            if (k > 0 && !mbar_test(&empty[s], (k - 1) & 1)) return;
            const bool down = l < a->L && ph == 3;
            const int K = down ? a->I : a->H;
            const int n = min(down ? a->rows_i : a->rows_h, r1 - r);
            const __half* W = l == a->L ? a->Wlm
                              : ph == 0 ? a->layers[l].wqkv
                              : ph == 1 ? a->layers[l].wo
                              : ph == 2 ? a->layers[l].wgu
                                        : a->layers[l].wd;
            const unsigned bytes = (unsigned)n * K * 2;
            mbar_expect_tx(&full[s], bytes);
            bulk_g2s(ring + (size_t)s * kPersistStage, W + (size_t)r * K, bytes, &full[s]);
            r += n;
            ++issued;
        }
    }
    // Feed the whole sequence, waiting (bounded) for each stage to be
    // released; false if a wait gave up.
    __device__ __forceinline__ bool run() {
        while (!done) {
            refill();
            if (done) break;
            const int s = issued % a->stages;
            const unsigned k = issued / a->stages;
            const u64 t0 = now_ns();
            while (!mbar_test(&empty[s], (k - 1) & 1)) {
                if (now_ns() - t0 > wait_limit()) return false;
                __nanosleep(20);
            }
        }
        return true;
    }
    // Before leaving early: wait (bounded) for the copies still in flight.
    __device__ __forceinline__ void drain() {
        for (int j = max(0, issued - a->stages); j < issued; ++j) {
            const u64 t0 = now_ns();
            while (!mbar_try_wait(&full[j % a->stages], (j / a->stages) & 1) && now_ns() - t0 < wait_limit()) {
            }
        }
    }
};

// Write one value to all copies of a buffer (`stride` packets apart).
__device__ __forceinline__ void pk_put_all(u64* p, int stride, float v, unsigned ep) {
#pragma unroll
    for (int r = 0; r < kPkRep; ++r) pk_put(p + (size_t)r * stride, v, ep);
}

// The kernel's dynamic shared memory, named at file scope so that the
// out-of-line helpers below derive their pointers from a shared-memory
// object (a generic pointer passed in leaves the compiler generic loads).
// Layout: the weight ring (kPersistStages stages), then the mbarriers and
// the reduction scratch (256 bytes), then the activation area (kActOff).
extern __shared__ __align__(128) unsigned char persist_smem[];
constexpr int kActOff = kPersistStages * kPersistStage + 256;

__device__ __forceinline__ float* act_smem() { return reinterpret_cast<float*>(persist_smem + kActOff); }
__device__ __forceinline__ const __half* stage_smem(int s) {
    return reinterpret_cast<const __half*>(persist_smem + (size_t)s * kPersistStage);
}
__device__ __forceinline__ uint64_t* full_bars() { return reinterpret_cast<uint64_t*>(persist_smem + kPersistStages * kPersistStage); }

// One lane's share of an activation vector of K floats as the canonical
// row dot reads it (rowdot.cuh): chunks c = lane + 32 u of eight floats,
// held in registers so that a warp reading many rows loads x once.
template <int K>
struct XLane {
    static constexpr int kC = K / 8, kP = (kC + 31) / 32;
    float4 a[kP], b[kP];
    __device__ __forceinline__ void load(const float* xs) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int u = 0; u < kP; ++u) {
            const int c = lane + 32 * u;
            if (c < kC) {
                a[u] = *reinterpret_cast<const float4*>(xs + c * 8);
                b[u] = *reinterpret_cast<const float4*>(xs + c * 8 + 4);
            } else {
                a[u] = b[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
};

// The canonical row dot of R rows (in shared memory) with x in registers:
// lane l adds chunks l, l + 32, ... in that order into four partial sums
// per row, then the xor butterfly -- warp_rows_dot's operations in its
// order, so the same bits.
template <int K, int R>
__device__ __forceinline__ void rows_dot_x(const __half* const (&rows)[R], const XLane<K>& x, float (&acc)[R]) {
    constexpr int kC = XLane<K>::kC, kP = XLane<K>::kP;
    const int lane = threadIdx.x & 31;
    Acc4 part[R];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) part[r].a[e] = 0.f;
    uint4 wv[R][kP];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int u = 0; u < kP; ++u) {
            const int c = lane + 32 * u;
            wv[r][u] = c < kC ? *reinterpret_cast<const uint4*>(rows[r] + (size_t)c * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
    for (int u = 0; u < kP; ++u)
        if (lane + 32 * u < kC)
#pragma unroll
            for (int r = 0; r < R; ++r) dot8_f16_4(wv[r][u], x.a[u], x.b[u], part[r]);
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = warp_sum(dot4_total(part[r]));
}

// Wait (bounded) for an mbarrier phase.
__device__ __forceinline__ bool wait_bar(uint64_t* b, unsigned par) {
    if (mbar_try_wait(b, par)) return true;
    const u64 t0 = now_ns();
    while (now_ns() - t0 < wait_limit())
        if (mbar_try_wait(b, par)) return true;
    return false;
}

// Dot products of this warp's row pairs of a slice of nrows rows whose
// chunks (sixteen rows each) sit in the ring from position it0 on: rows
// (2w, 2w + 1) of each chunk, against the activation vector at the start of
// the activation area.  Pair i's two sums go to res[2i], res[2i + 1] (lane
// 0).  Each warp waits for a chunk's stage only when it reads it and
// releases it (one of the stage's eight arrivals) as soon as its dot is
// done, so the ring refills while the slice is still being computed.
// Returns false if a wait gave up (the stages are still released).
// Compiled as a function of its own with K known: inside the large kernel
// body the same loop ran several times slower.
template <int K>
__device__ __noinline__ bool warp_stage_pairs(int it0, int nrows, float* res) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* full = full_bars();
    uint64_t* empty = full + kPersistStages;
    XLane<K> x;
    x.load(act_smem());
    bool ok = true;
    const int nch = (nrows + 15) / 16;
    int i = 0;
    // Two stages at a time where this warp has a full pair in both: the
    // four rows' loads and reductions overlap (each row's own operations and
    // their order are unchanged).
    for (; i + 1 < nch && 16 * (i + 1) + 2 * warp + 1 < nrows; i += 2) {
        const int itA = it0 + i, sA = itA % kPersistStages;
        const int itB = itA + 1, sB = itB % kPersistStages;
        if (ok && !wait_bar(&full[sA], (unsigned)(itA / kPersistStages) & 1u)) ok = false;
        if (ok && !wait_bar(&full[sB], (unsigned)(itB / kPersistStages) & 1u)) ok = false;
        if (ok) {
            const __half* stA = stage_smem(sA);
            const __half* stB = stage_smem(sB);
            const __half* rows[4] = {stA + (size_t)(2 * warp) * K, stA + (size_t)(2 * warp + 1) * K,
                                     stB + (size_t)(2 * warp) * K, stB + (size_t)(2 * warp + 1) * K};
            float acc[4];
            rows_dot_x<K, 4>(rows, x, acc);
            if (lane == 0) {
                res[2 * i] = acc[0];
                res[2 * i + 1] = acc[1];
                res[2 * i + 2] = acc[2];
                res[2 * i + 3] = acc[3];
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&empty[sA]);
            mbar_arrive(&empty[sB]);
        }
    }
    for (; i < nch; ++i) {
        const int it = it0 + i, s = it % kPersistStages;
        if (16 * i + 2 * warp < nrows) {
            if (ok && !wait_bar(&full[s], (unsigned)(it / kPersistStages) & 1u)) ok = false;
            if (ok) {
                const __half* st = stage_smem(s);
                const bool two = 16 * i + 2 * warp + 1 < nrows;
                const __half* rows[2] = {st + (size_t)(2 * warp) * K,
                                         st + (size_t)(two ? 2 * warp + 1 : 2 * warp) * K};
                float acc[2];
                rows_dot_x<K, 2>(rows, x, acc);
                if (lane == 0) {
                    res[2 * i] = acc[0];
                    res[2 * i + 1] = acc[1];
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    __syncwarp();
    return ok;
}

// An activation vector of K floats stored as two half arrays: floats
// 0..3 of each 8-float chunk c at xa[4c..4c+3], floats 4..7 at
// xh[4c..4c+3] (xh = xa + K/2), so a warp reading chunk c = lane + 32 u
// reads 16 consecutive bytes per lane from each half: no bank conflicts,
// where the plain layout (32-byte lane stride) conflicts two ways.
__device__ __forceinline__ int split_half_index(int j, int half) {
    return ((j & 7) < 4 ? 0 : half) + (j >> 3) * 4 + (j & 3);
}

// The canonical row dot (lane l adds chunks l, l + 32, ... in order into
// four partial sums, then the xor butterfly) of one shared-memory row with
// x in the split-half layout, U chunks of loads in flight per lane: the
// operations and order of warp_rows_dot, so the same bits.
template <int K, int U>
__device__ __forceinline__ float row_dot_split(const __half* row, const float* xa, const float* xh) {
    constexpr int kC = K / 8;
    const int lane = threadIdx.x & 31;
    Acc4 part;
#pragma unroll
    for (int e = 0; e < 4; ++e) part.a[e] = 0.f;
    for (int i0 = 0; i0 * 32 < kC; i0 += U) {
        uint4 wv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = lane + 32 * (i0 + u);
            wv[u] = c < kC ? *reinterpret_cast<const uint4*>(row + (size_t)c * 8) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = lane + 32 * (i0 + u);
            if (c < kC)
                dot8_f16_4(wv[u], *reinterpret_cast<const float4*>(xa + 4 * c),
                           *reinterpret_cast<const float4*>(xh + 4 * c), part);
        }
    }
    return warp_sum(dot4_total(part));
}

// Dot products of this warp's rows q = w, w + 8, ... of a slice of nrows
// rows of K stored rpc to a chunk, the chunks in the ring from position it0
// on, against the activation vector in the split-half layout; row k's sum
// goes to res[k].  Waits and releases per stage as warp_stage_pairs does.
template <int K>
__device__ __noinline__ bool warp_stage_rows(int it0, int rpc, int nrows, float* res) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* full = full_bars();
    uint64_t* empty = full + kPersistStages;
    const float* xa = act_smem();
    const float* xh = xa + K / 2;
    bool ok = true;
    const int nch = (nrows + rpc - 1) / rpc;
    int k = 0;
    for (int j = 0; j < nch; ++j) {
        const int it = it0 + j, s = it % kPersistStages;
        for (int q = j * rpc; q < min(nrows, (j + 1) * rpc); ++q) {
            if ((q & 7) != warp) continue;
            if (ok && !wait_bar(&full[s], (unsigned)(it / kPersistStages) & 1u)) ok = false;
            if (ok) {
                const float v = row_dot_split<K, 8>(stage_smem(s) + (size_t)(q - j * rpc) * K, xa, xh);
                if (lane == 0) res[k] = v;
            }
            ++k;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    __syncwarp();
    return ok;
}

// The tied LM head over this CTA's vocabulary rows [r0, r1): chunks of 16
// rows stream through the ring from ring position it0; the final-normed
// hidden state (activation area) is held in registers for the whole slice.
// Warp w takes rows 2w, 2w + 1 of each chunk; lane 0 stores the logits (if
// asked) and keeps the warp's running argmax (lowest index on ties).
// Returns false if a wait gave up (the stages are still released).
template <int K>
__device__ __noinline__ bool lm_head_rows(int it0, int r0, int r1, float* logits, float* best_v, int* best_i) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t* full = full_bars();
    uint64_t* empty = full + kPersistStages;
    XLane<K> x;
    x.load(act_smem());
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    bool ok = true;
    int it = it0;
    for (int r = r0; r < r1; r += 16, ++it) {
        const int n = min(16, r1 - r);
        const int s = it % kPersistStages;
        if (ok && !wait_bar(&full[s], (unsigned)(it / kPersistStages) & 1u)) ok = false;
        if (ok && 2 * warp < n) {
            const __half* st = stage_smem(s);
            const bool two = 2 * warp + 1 < n;
            const __half* rows[2] = {st + (size_t)(2 * warp) * K, st + (size_t)(two ? 2 * warp + 1 : 2 * warp) * K};
            float acc[2];
            rows_dot_x<K, 2>(rows, x, acc);
            if (lane == 0) {
                const int row = r + 2 * warp;
                if (logits) {
                    logits[row] = acc[0];
                    if (two) logits[row + 1] = acc[1];
                }
                argmax_merge(bv, bi, acc[0], row);
                if (two) argmax_merge(bv, bi, acc[1], row + 1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    *best_v = bv;
    *best_i = bi;
    return ok;
}

// One attention chunk (keys, values and queries already in the attention
// area) for `group` query heads of one kv head (all of its heads, or a
// subset); writes each head's partial (m, l, acc[64]) to packet copy 0
// (only the head's merging CTA reads it): head h's partial at
// out + h * head_stride.
__device__ __noinline__ void attn_unit_compute(int group, int nj, u64* out, int head_stride, unsigned ep) {
    AttnSmem& at = *reinterpret_cast<AttnSmem*>(act_smem());
    attn_chunk<SyncCompute>(at, group, nj, [&](int h, int d, float acc, float m, float lsum) {
        u64* pr = out + (size_t)h * head_stride;
        pk_put(pr + 2 + d, acc, ep);
        if (d == 0) {
            pk_put(pr, m, ep);
            pk_put(pr + 1, lsum, ep);
        }
    });
}

// Merge of one head: gather its n_chunks partials into the activation
// area at float offset stg_off,
// merge them with the attn_merge arithmetic (chunk order) and publish the
// 64 outputs to every packet copy of dst.  A function of its own so that
// the main loop's code generation does not change with it.
__device__ __noinline__ void merge_head(PkReader& rd, const u64* att_h, int n_chunks, int stg_off, u64* dst,
                                        int copy_stride, unsigned ep) {
    float* stg = act_smem() + stg_off;
    pk_gather<8>(rd, n_chunks * kPartStride, [&](int j) { return att_h + j; }, [&](int j, float v) { stg[j] = v; },
                 [] {});
    SyncCompute::sync();
    const int tid = threadIdx.x;
    if (tid < kHd) {
        const float ov = attn_merge(n_chunks, tid, [&](int cc, int i) { return stg[cc * kPartStride + i]; });
        pk_put_all(dst + tid, copy_stride, ov, ep);
    }
}

template <int HC, int IC>
__global__ void __launch_bounds__(kThreads, 1) k_decode_persistent(PersistentArgs a) {
    unsigned char* ring = persist_smem;
    uint64_t* full = full_bars();
    uint64_t* empty = full + kPersistStages;
    float* red = reinterpret_cast<float*>(empty + kPersistStages);
    float* act = act_smem();
    float* xr = act + a.act_floats;  // raw x [H]
    AttnSmem& at = *reinterpret_cast<AttnSmem*>(act);
    float* xs = act;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, G = gridDim.x;
    constexpr int H = HC, I = IC;
    const int V = a.V, L = a.L, nh = a.nh, nkv = a.nkv;
    const int group = nh / nkv;
    const int np = a.nqkv / 2;
    const int rpc_i = a.rows_i;

    if (tid == 0) {
        wait_limit_s = a.wait_ns;
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCompute / 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const unsigned ep = *a.epoch + 1;
    const int p = a.pos[0], t = a.tok[0], slot = a.slot[0];
    if (p < 0 || p >= a.n_ctx || t < 0 || t >= V || slot < 0 || slot >= a.max_seqs) {
        if (tid == 0 && c == 0) raise_guard(a.err, (p < 0 || p >= a.n_ctx) ? kGuardPosition : kGuardToken);
        return;
    }
    const int n_chunks = (p + 1 + kAttCh - 1) / kAttCh;
    const PkLayout lay(a.nqkv, H, I, nh, a.max_chunks);

    if (warp >= kCompute / 32) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegFeed));
        if (tid != kCompute) return;
        Feeder feed;
        feed.init(&a, ring, full, empty, c, G);
        if (!feed.run()) raise_guard(a.err, kGuardTimeout);
        feed.drain();
        return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegCompute));

    // ------------------------------------------------------------------
    // Compute warps.  Every load that does not depend on the incoming
    // activations (norm weights, biases, RoPE factors, cached keys/values)
    // is issued before the wait for them.
    // ------------------------------------------------------------------
    PkReader rd{ep};
    int it = 0;
    bool dead = false, bad = false;
    // Profiling marks (QWEN2_FLAG_PROFILE): mark(id) stores the global timer
    // at slot id; per layer l the slots are 1 + 16 l + k (see kMark*).
    auto mark = [&](int id) {
        if (a.prof && tid == 0) a.prof[(size_t)c * a.prof_marks + id] = (long long)now_ns();
    };
    mark(0);
    auto idle = [&]() {};
    __shared__ float res_s[8][16];  // per-warp dot results of the current phase
    float* res = res_s[warp];
    // Stream this CTA's slice [r0, r1) of a K = H matrix (sixteen rows to a
    // ring stage) through warp_stage_pairs, then epi(first row, rows) on the
    // results in res.  A slice of more stages than res holds pairs for a
    // warp goes one stage per call.  A wait that gives up marks the thread
    // bad (the epilogue is skipped); the phase end turns that into a
    // group-wide decision.
    auto stream_pairs = [&](int r0, int r1, auto&& epi) {
        const int nch = (r1 - r0 + 15) / 16;
        const int per = nch <= 8 ? nch : 1;
        for (int j = 0; j < nch; j += per) {
            const int rr = r0 + 16 * j, nn = min(16 * per, r1 - rr);
            if (warp_stage_pairs<H>(it + j, nn, res)) epi(rr, nn);
            else bad = true;
        }
        it += nch;
    };
    // The same for the K = I slice of down_proj, rpc rows to a stage.
    auto stream_rows = [&](int r0, int r1, int rpc, auto&& epi) {
        const int nch = (r1 - r0 + rpc - 1) / rpc;
        const int per = (r1 - r0) <= 8 * 16 ? nch : 1;
        for (int j = 0; j < nch; j += per) {
            const int rr = r0 + rpc * j, nn = min(rpc * per, r1 - rr);
            if (warp_stage_rows<I>(it + j, rpc, nn, res)) epi(rr, nn);
            else bad = true;
        }
        it += nch;
    };
    auto phase_end = [&]() {
        dead = compute_any(bad || rd.failed);
        return dead;
    };
    // Arrive at / wait for counter `k` of this launch (thread 0 of the group).
    auto arrive = [&](int k) {
        if (tid == 0) cnt_arrive(a.cnt + (size_t)k * kCntStride);
    };
    auto wait_cnt = [&](int k) {
        if (tid == 0) {
            const u64* cp = a.cnt + (size_t)k * kCntStride;
            const u64 target = (u64)ep * (u64)G;
            if (pk_raw(cp) < target) {
                const u64 t0 = now_ns();
                while (pk_raw(cp) < target) {
                    if (now_ns() - t0 > wait_limit()) {
                        bad = true;
                        break;
                    }
                    __nanosleep(20);
                }
            }
        }
        SyncCompute::sync();
    };
    auto gather = [&](const u64* src, int n, float* dst) {
        pk_gather<8>(rd, n, [&](int j) { return src + j; }, [&](int j, float v) { dst[j] = v; }, idle);
    };
    // Norm weights of the next normalisation, in registers (j = tid + 256 k).
    float nw[4];
    auto load_norm = [&](const float* w) {
#pragma unroll
        for (int k = 0; k < 4; ++k) nw[k] = tid + 256 * k < H ? w[tid + 256 * k] : 0.f;
    };
    // RMSNorm of xr into xs with the prefetched weights; the same arithmetic
    // as norm_rows_to_smem (per-thread sum in index order, block_sum).
    auto norm = [&]() {
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (tid + 256 * k < H) ss = fmaf(xr[tid + 256 * k], xr[tid + 256 * k], ss);
        const float sc = rms_scale(block_sum<SyncCompute>(ss, red), H, a.eps);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (tid + 256 * k < H) xs[tid + 256 * k] = __fmul_rn(__fmul_rn(xr[tid + 256 * k], sc), nw[k]);
        SyncCompute::sync();
    };

    const size_t head_stride = (size_t)a.n_ctx * kHd;
    // This CTA's row ranges, the same for every layer.
    const int qkv_r0 = 2 * split(np, c, G), qkv_r1 = 2 * split(np, c + 1, G);
    const int o_r0 = 2 * split(H / 2, c, G), o_r1 = 2 * split(H / 2, c + 1, G);
    const int gu_r0 = 2 * split(I, c, G), gu_r1 = 2 * split(I, c + 1, G);
    const int d_r0 = split(H, c, G), d_r1 = split(H, c + 1, G);
    const int rc = c % kPkRep;  // the packet copy this CTA reads
    for (int l = 0; l < L && !dead; ++l) {
        const PersistLayer& Lw = a.layers[l];
        u64* pk = a.pk + (size_t)l * lay.per_layer;
        const u64* pk_prev = a.pk + (size_t)(l - 1) * lay.per_layer;
        const size_t cache0 = ((size_t)slot * L + l) * 2 * nkv;

        // ---- RMSNorm + Q/K/V + bias + RoPE + KV store -----------------
        load_norm(Lw.attn_norm);
        // Bias and RoPE factors of this warp's first pair, loaded now so the
        // epilogue does not wait for them.
        float pb0 = 0.f, pb1 = 0.f;
        float2 pcs = make_float2(1.f, 0.f);
        if (lane == 0 && qkv_r0 + 2 * warp < qkv_r1) {
            const int pr = qkv_r0 + 2 * warp;
            pb0 = Lw.bqkv[pr];
            pb1 = Lw.bqkv[pr + 1];
            pcs = a.rope[(size_t)p * (kHd / 2) + ((pr % kHd) >> 1)];
        }
        if (l == 0) {
            for (int j = tid; j < H; j += kCompute) xr[j] = __half2float(a.E[(size_t)t * H + j]);
        } else {
            gather(pk_prev + lay.x2 + (size_t)rc * lay.n_x, H, xr);
        }
        if (phase_end()) break;
        const int mb = 1 + 16 * l;
        mark(mb + 0);
        norm();
        mark(mb + 1);
        // Sixteen rows per stage, one row pair per warp: warp w takes rows
        // 2w, 2w + 1 of each stage of its slice.
        stream_pairs(qkv_r0, qkv_r1, [&](int r0_, int n_) {
            for (int q = warp, i = 0; 2 * q < n_; q += 8, ++i) {
                const int pr = r0_ + 2 * q;  // packed row of the pair
                const float acc[2][1] = {{res[2 * i]}, {res[2 * i + 1]}};
                if (lane == 0) {
                    const int s = pr / kHd, i = (pr % kHd) >> 1;
                    const bool first = pr == qkv_r0 + 2 * warp;
                    const float b0 = first ? pb0 : Lw.bqkv[pr];
                    const float b1 = first ? pb1 : Lw.bqkv[pr + 1];
                    const float v0 = acc[0][0] + b0, v1 = acc[1][0] + b1;
                    if (s < nh + nkv) {
                        const float2 cs = first ? pcs : a.rope[(size_t)p * (kHd / 2) + i];
                        float ra, rb;
                        rope_pair(v0, v1, cs, ra, rb);
                        pk_put(pk + lay.qkv + s * kHd + i, ra, ep);
                        pk_put(pk + lay.qkv + s * kHd + i + kHd / 2, rb, ep);
                        if (s >= nh) {
                            float* kr = a.kv + (cache0 + (s - nh)) * head_stride + (size_t)p * kHd;
                            kr[i] = ra;
                            kr[i + kHd / 2] = rb;
                        }
                    } else {
                        pk_put(pk + lay.qkv + s * kHd + i, v0, ep);
                        pk_put(pk + lay.qkv + s * kHd + i + kHd / 2, v1, ep);
                        float* vr = a.kv + (cache0 + nkv + (s - nh - nkv)) * head_stride + (size_t)p * kHd;
                        vr[i] = v0;
                        vr[i + kHd / 2] = v1;
                    }
                }
            }
        });
        if (phase_end()) break;
        arrive(l * 5 + 0);
        mark(mb + 2);
        if (a.test_stall && l == 0) {
            // Test hook: wait on a counter no CTA arrives at.  The wait runs
            // out (a shortened limit), the CTAs leave, and the guard word
            // reports it.
            wait_cnt(L * 5 + 1);
            if (phase_end()) break;
        }

        // ---- attention: units (kv head g, chunk of 64 keys, query heads) -
        // When there are fewer (kv head, chunk) pairs than CTAs, each pair's
        // query heads are split into hsplit subsets on different CTAs: a
        // head's scores, softmax and sums do not depend on the other heads
        // of its group, so the partials are the same bits, computed by up
        // to `group` times more SMs.
        bool qkv_seen = false;
        const int hsplit = max(1, min(group, G / (nkv * n_chunks)));
        for (int u = c; u < nkv * n_chunks * hsplit; u += G) {
            const int sub = u % hsplit, gu_ = u / hsplit;
            const int g = gu_ / n_chunks, ch = gu_ % n_chunks;
            const int h0 = sub * group / hsplit, hn = (sub + 1) * group / hsplit - h0;
            const int j0 = ch * kAttCh, nj = min(kAttCh, p + 1 - j0);
            const int nold = min(nj, p - j0);  // keys of earlier steps, read from the cache
            const float* kb = a.kv + (cache0 + g) * head_stride + (size_t)j0 * kHd;
            const float* vb = a.kv + (cache0 + nkv + g) * head_stride + (size_t)j0 * kHd;
            float4 kk[4], vv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = tid + 256 * k, j = e / (kHd / 4), d4 = (e % (kHd / 4)) * 4;
                if (j < nold) {
                    kk[k] = __ldcg(reinterpret_cast<const float4*>(kb + (size_t)j * kHd + d4));
                    vv[k] = __ldcg(reinterpret_cast<const float4*>(vb + (size_t)j * kHd + d4));
                }
            }
            SyncCompute::sync();  // the previous unit is done with `at`
            if (!qkv_seen) {
                // q, k and v are read as epoch-tagged packets (a unit re-polls
                // the ones not yet written): no arrival counter to wait for,
                // which would add an L2 round trip.
                qkv_seen = true;
                mark(mb + 3);
            }
            const u64* qp = pk + lay.qkv + (size_t)(g * group + h0) * kHd;
            pk_gather<2>(rd, hn * kHd, [&](int e) { return qp + e; },
                         [&](int e, float v) { at.q[e / kHd][e % kHd] = v; }, idle);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int e = tid + 256 * k, j = e / (kHd / 4), d4 = (e % (kHd / 4)) * 4;
                if (j < nold) {
                    at.k[j][d4] = kk[k].x;
                    at.k[j][d4 + 1] = kk[k].y;
                    at.k[j][d4 + 2] = kk[k].z;
                    at.k[j][d4 + 3] = kk[k].w;
                    *reinterpret_cast<float4*>(&at.v[j][d4]) = vv[k];
                }
            }
            if (nold < nj) {  // this step's key and value (position p): from the packets
                const u64* kp = pk + lay.qkv + (size_t)(nh + g) * kHd;
                const u64* vp = pk + lay.qkv + (size_t)(nh + nkv + g) * kHd;
                pk_gather<1>(rd, 2 * kHd, [&](int e) { return e < kHd ? kp + e : vp + (e - kHd); },
                             [&](int e, float v) {
                                 if (e < kHd) at.k[nold][e] = v;
                                 else at.v[nold][e - kHd] = v;
                             }, idle);
            }
            SyncCompute::sync();
            attn_unit_compute(hn, nj,
                              pk + lay.att + ((size_t)(g * group + h0) * a.max_chunks + ch) * kPartStride,
                              a.max_chunks * kPartStride, ep);
        }
        if (phase_end()) break;
        arrive(l * 5 + 1);
        mark(mb + 4);

        // ---- attention output, o_proj + residual -------------------------
        // CTA h (h < nh) merges head h's chunk partials (the attn_merge
        // arithmetic, in chunk order) and publishes o_h; every CTA gathers
        // all of o.  Two short L2 round trips on the critical path instead
        // of every CTA gathering and merging every partial.
        {
            const u64* att = pk + lay.att;  // partials: copy 0 only
            u64* ob = a.pk + lay.o_base(L, G, l);
            // The merging CTA polls the partials' packets by epoch directly.
            mark(mb + 5);
            if (c < nh)
                merge_head(rd, att + (size_t)c * a.max_chunks * kPartStride, n_chunks, H, ob + (size_t)c * kHd,
                           lay.n_o, ep);
            gather(ob + (size_t)rc * lay.n_o, nh * kHd, xs);
            if (phase_end()) break;
        }
        mark(mb + 6);
        stream_pairs(o_r0, o_r1, [&](int r0_, int n_) {
            for (int q = warp, i = 0; 2 * q < n_; q += 8, ++i) {
                const int r = r0_ + 2 * q;
                // xr still holds this layer's input x (gathered for Q/K/V);
                // lanes 0-7 write copy (lane % 4) of row r + lane / 4.
                if (lane < 2 * kPkRep) {
                    const int e = lane / kPkRep, k = lane % kPkRep;
                    pk_put(pk + lay.x1 + (size_t)k * lay.n_x + r + e, xr[r + e] + res[2 * i + e], ep);
                }
            }
        });
        load_norm(Lw.ffn_norm);
        if (phase_end()) break;
        arrive(l * 5 + 2);
        mark(mb + 7);

        // ---- RMSNorm + gate/up + SiLU(gate) * up ----------------------
        // The packets carry the epoch: gather them directly (a thread
        // re-polls the ones not yet written) instead of first waiting for
        // the phase's arrival counter, which would add an L2 round trip.
        mark(mb + 8);
        gather(pk + lay.x1 + (size_t)rc * lay.n_x, H, xr);
        if (phase_end()) break;
        mark(mb + 9);
        norm();
        // Pair (gate j, up j) in rows 2j, 2j + 1; one pair per warp per stage.
        // Lane 4i + k writes copy k of pair i's output, element j of m stored
        // at its split-half position, the layout down_proj reads.
        auto gu_out = [&](int r0, int n) {
            const int i = lane / kPkRep, k = lane % kPkRep, q = warp + 8 * i;
            if (i < 32 / kPkRep && 2 * q < n)
                pk_put(pk + lay.m + (size_t)k * lay.n_m + split_half_index((r0 + 2 * q) >> 1, I / 2),
                       silu_f(res[2 * i]) * res[2 * i + 1], ep);
        };
        stream_pairs(gu_r0, gu_r1, gu_out);
        if (phase_end()) break;
        arrive(l * 5 + 3);
        mark(mb + 10);

        // ---- down + residual ------------------------------------------
        // SiLU(gate) * up is a large gather (I packets): poll the counter
        // first rather than have every thread re-poll packets.
        wait_cnt(l * 5 + 3);
        mark(mb + 11);
        const u64* mp = pk + lay.m + (size_t)rc * lay.n_m;
        pk_gather<20>(rd, I, [&](int j) { return mp + j; }, [&](int j, float v) { xs[j] = v; }, idle);
        if (phase_end()) break;
        mark(mb + 12);
        // xr holds x after the attention add (gathered for gate/up).
        auto down_out = [&](int r0, int n) {
            const int i = lane / kPkRep, k = lane % kPkRep, q = warp + 8 * i;
            if (i < 32 / kPkRep && q < n) pk_put(pk + lay.x2 + (size_t)k * lay.n_x + r0 + q, xr[r0 + q] + res[i], ep);
        };
        stream_rows(d_r0, d_r1, rpc_i, down_out);
        if (phase_end()) break;
        arrive(l * 5 + 4);
        mark(mb + 13);
    }

    // ---- final RMSNorm + tied LM head + argmax --------------------------
    __shared__ float wv_s[8];
    __shared__ int wi_s[8];
    float best_v = -INFINITY;
    int best_i = 0x7fffffff;
    if (!dead) {
        load_norm(a.final_norm);
        wait_cnt((L - 1) * 5 + 4);
        gather(a.pk + (size_t)(L - 1) * lay.per_layer + lay.x2 + (size_t)rc * lay.n_x, H, xr);
        phase_end();
        mark(1 + 16 * L);
    }
    if (!dead) {
        norm();
        if (c == 0)
            for (int j = tid; j < H; j += kCompute) a.hidden[j] = xs[j];
        const int v0 = split(V, c, G), v1 = split(V, c + 1, G);
        float bv;
        int bi;
        if (!lm_head_rows<H>(it, v0, v1, a.logits, &bv, &bi)) bad = true;
        best_v = bv;
        best_i = bi;
        it += (v1 - v0 + 15) / 16;
        phase_end();
    }
    if (!dead) {
        mark(2 + 16 * L);
        if (lane == 0) {
            wv_s[warp] = best_v;
            wi_s[warp] = best_i;
        }
        SyncCompute::sync();
        u64* am = a.pk + (size_t)L * lay.per_layer;
        if (tid == 0) {
            float v = wv_s[0];
            int i = wi_s[0];
            for (int w = 1; w < 8; ++w) argmax_merge(v, i, wv_s[w], wi_s[w]);
            pk_put(am + 2 * c, v, ep);
            pk_put(am + 2 * c + 1, __int_as_float(i), ep);
        }
        arrive(L * 5);
        if (c == 0) {
            // Stage 2: merge the per-CTA pairs; the id becomes the next token.
            wait_cnt(L * 5);
            float v = -INFINITY;
            int i = 0x7fffffff;
            for (int k = tid; k < G; k += kCompute) {
                const float kv_ = rd.get(am + 2 * k);
                argmax_merge(v, i, kv_, __float_as_int(rd.get(am + 2 * k + 1)));
            }
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, v, o);
                const int oi = __shfl_xor_sync(0xffffffffu, i, o);
                argmax_merge(v, i, ov, oi);
            }
            SyncCompute::sync();
            if (lane == 0) {
                wv_s[warp] = v;
                wi_s[warp] = i;
            }
            const bool failed = compute_any(rd.failed);
            if (tid == 0 && !failed) {
                float fv = wv_s[0];
                int fi = wi_s[0];
                for (int w = 1; w < 8; ++w) argmax_merge(fv, fi, wv_s[w], wi_s[w]);
                if (fi < 0 || fi >= V) {
                    raise_guard(a.err, kGuardShape);
                    fi = 0;
                }
                a.ids_hist[(size_t)(*a.step % kIdsHist) * a.hist_stride] = fi;
                a.tok[0] = fi;
                a.pos[0] = p + 1;
                *a.step = *a.step + 1;
                *a.epoch = ep;
            }
            if (failed) dead = true;
        }
        mark(3 + 16 * L);
    }
    if (dead && tid == 0) raise_guard(a.err, kGuardTimeout);
}

namespace {
// The shapes the persistent kernel is instantiated for (hidden, intermediate).
typedef void (*PersistKernel)(PersistentArgs);
PersistKernel pick_kernel(int H, int I) {
    if (H == 896 && I == 4864) return k_decode_persistent<896, 4864>;  // Qwen2.5-0.5B
    if (H == 256 && I == 1024) return k_decode_persistent<256, 1024>;
    if (H == 384 && I == 640) return k_decode_persistent<384, 640>;
    return nullptr;
}
}  // namespace

cudaError_t persistent_setup(Ctx& c) {
    const qwen2_config& g = c.cfg;
    const int H = g.hidden, I = g.intermediate;
    c.pers.ok = false;
    if (g.weight_format != QWEN2_WEIGHTS_F16) {
        c.pers.why_not = "the persistent kernel streams f16 weights only";
        return cudaSuccess;
    }
    if (g.head_dim != kHd) {
        c.pers.why_not = "the persistent kernel is built for head_dim 64";
        return cudaSuccess;
    }
    const size_t act = std::max(sizeof(AttnSmem), (size_t)std::max(H, I) * 4);
    const size_t smem = (size_t)kPersistStages * kPersistStage + 256 + act + (size_t)H * 4;
    int dev_max = 0;
    cudaDeviceGetAttribute(&dev_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, c.device);
    // Sixteen rows of K = H per stage (one row pair per compute warp).
    const int rows_h = 2 * H * 16 <= kPersistStage ? 16 : 0;
    const int rows_i = kPersistStage / (2 * I);
    const int max_qkv_rows = 2 * ((c.nqkv / 2 + c.n_sm - 1) / c.n_sm), max_o_rows = 2 * ((H / 2 + c.n_sm - 1) / c.n_sm);
    if (smem + 1024 > (size_t)dev_max || rows_h < 2 || rows_i < 1 ||
        max_qkv_rows > rows_h * kPersistStages || max_o_rows > rows_h * kPersistStages) {
        c.pers.why_not = "shared memory or stage size does not fit this shape";
        return cudaSuccess;
    }
    const PersistKernel kern = pick_kernel(H, I);
    if (!kern) {
        c.pers.why_not = "no persistent kernel instantiated for hidden " + std::to_string(H) + ", intermediate " +
                         std::to_string(I);
        return cudaSuccess;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) {
        c.pers.why_not = "occupancy query gives 0 blocks per SM";
        return cudaSuccess;
    }
    int coop = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c.device);
    if (!coop) {
        c.pers.why_not = "device has no cooperative launch";
        return cudaSuccess;
    }
    c.pers.grid = c.n_sm;
    c.pers.kernel = reinterpret_cast<const void*>(kern);
    c.pers.smem = smem;
    c.pers.rows_h = rows_h;
    c.pers.rows_i = rows_i;
    c.pers.act_floats = (int)(act / 4);
    c.pers.max_chunks = (g.n_ctx + kAttCh - 1) / kAttCh;
    // Chunk-merge staging after o [H]: all heads' partials at short
    // context, one head's partials (the per-head merge) at long context.
    c.pers.merge_group = 0;
    if (c.pers.max_chunks * kPartStride > c.pers.act_floats - H || g.n_head * kHd > 1024 ||
        g.n_head > c.pers.grid) {
        c.pers.why_not = "attention merge staging does not fit (n_ctx or heads too large)";
        return cudaSuccess;
    }
    const PkLayout lay(c.nqkv, H, I, g.n_head, c.pers.max_chunks);
    const size_t n_pk = lay.o_base(g.n_layer, c.pers.grid, g.n_layer);
    std::vector<PersistLayer> hl(g.n_layer);
    for (int l = 0; l < g.n_layer; ++l) {
        const DevLayer& D = c.layers[l];
        hl[l] = PersistLayer{D.wqkv.w, D.wo.w, D.wgu.w, D.wd.w, D.bqkv, D.attn_norm, D.ffn_norm};
    }
    void* p = nullptr;
    if ((e = cudaMalloc(&p, hl.size() * sizeof(PersistLayer))) != cudaSuccess) return e;
    c.allocs.push_back(p);
    c.pers.layers = static_cast<PersistLayer*>(p);
    if ((e = cudaMemcpy(p, hl.data(), hl.size() * sizeof(PersistLayer), cudaMemcpyHostToDevice)) != cudaSuccess)
        return e;
    if ((e = cudaMalloc(&p, n_pk * 8)) != cudaSuccess) return e;
    c.allocs.push_back(p);
    c.pers.pk = static_cast<unsigned long long*>(p);
    if ((e = cudaMemset(p, 0, n_pk * 8)) != cudaSuccess) return e;
    c.pers.pk_bytes = n_pk * 8;
    // One counter per phase of every layer, one for the argmax, and one
    // that nothing arrives at (the failure-detection test hook waits on it).
    c.pers.cnt_bytes = (size_t)(g.n_layer * 5 + 2) * kCntStride * 8;
    if ((e = cudaMalloc(&p, c.pers.cnt_bytes)) != cudaSuccess) return e;
    c.allocs.push_back(p);
    c.pers.cnt = static_cast<unsigned long long*>(p);
    if ((e = cudaMemset(p, 0, c.pers.cnt_bytes)) != cudaSuccess) return e;
    if ((e = cudaMalloc(&p, 4)) != cudaSuccess) return e;
    c.allocs.push_back(p);
    c.pers.epoch = static_cast<unsigned*>(p);
    if ((e = cudaMemset(p, 0, 4)) != cudaSuccess) return e;
    if (g.flags & QWEN2_FLAG_PROFILE) {
        c.pers.prof_marks = persistent_marks(g.n_layer);
        const size_t nb = (size_t)c.pers.grid * c.pers.prof_marks * 8;
        if ((e = cudaMalloc(&p, nb)) != cudaSuccess) return e;
        c.allocs.push_back(p);
        c.pers.prof = static_cast<long long*>(p);
        if ((e = cudaMemset(p, 0, nb)) != cudaSuccess) return e;
    }
    c.pers.ok = true;
    return cudaSuccess;
}

cudaError_t persistent_reset(Ctx& c) {
    if (!c.pers.ok) return cudaSuccess;
    cudaError_t e = cudaMemset(c.pers.pk, 0, c.pers.pk_bytes);
    if (e == cudaSuccess) e = cudaMemset(c.pers.cnt, 0, c.pers.cnt_bytes);
    if (e == cudaSuccess) e = cudaMemset(c.pers.epoch, 0, 4);
    return e;
}

cudaError_t enqueue_decode_persistent(Ctx& c, bool want_logits, cudaStream_t st) {
    PersistentArgs a;
    a.layers = c.pers.layers;
    a.E = c.embed.w;
    a.Wlm = c.lm_head.w;
    a.final_norm = c.final_norm;
    a.kv = c.kv;
    a.rope = c.rope;
    a.tok = c.ds.tok;
    a.pos = c.ds.pos;
    a.slot = c.ds.slot;
    a.step = c.ds.step;
    a.ids_hist = c.ds.ids_hist;
    a.hist_stride = c.cfg.max_seqs;
    a.epoch = c.pers.epoch;
    a.pk = c.pers.pk;
    a.logits = want_logits ? c.ws.logits : nullptr;
    a.hidden = c.ws.hidden;
    a.err = c.err;
    a.H = c.cfg.hidden;
    a.I = c.cfg.intermediate;
    a.V = c.cfg.vocab;
    a.L = c.cfg.n_layer;
    a.nh = c.cfg.n_head;
    a.nkv = c.cfg.n_kv_head;
    a.n_ctx = c.cfg.n_ctx;
    a.nqkv = c.nqkv;
    a.eps = c.cfg.rms_eps;
    a.stages = kPersistStages;
    a.rows_h = c.pers.rows_h;
    a.rows_i = c.pers.rows_i;
    a.act_floats = c.pers.act_floats;
    a.max_chunks = c.pers.max_chunks;
    a.max_seqs = c.cfg.max_seqs;
    a.merge_group = c.pers.merge_group;
    a.prof = c.pers.prof;
    a.cnt = c.pers.cnt;
    a.prof_marks = c.pers.prof_marks;
    a.wait_ns = c.pers.test_stall ? c.pers.test_wait_ns : kPersistWaitNs;
    a.test_stall = c.pers.test_stall;
    c.pers.test_stall = 0;  // one launch only
    if (c.pers.prof) {
        cudaError_t e = cudaMemsetAsync(c.pers.prof, 0, (size_t)c.pers.grid * c.pers.prof_marks * 8, st);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c.pers.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = c.pers.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, reinterpret_cast<PersistKernel>(c.pers.kernel), a);
}

}  // namespace qwen2
