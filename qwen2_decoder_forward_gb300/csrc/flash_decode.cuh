// Batched GQA decode attention over an f32 KV cache, for many sequences at
// ragged positions in one launch (flash-decoding with a persistent grid).
//
// What it computes (nnterp encyclopedia "qwen2", grouped-query attention;
// minfer "Qwen2 / Qwen2.5 Architecture Support", section 1): for every row b
// at position p_b and every query head h with kv head g = h / group,
//   s_j = q_h . K_j / sqrt(64)  (j = 0..p_b),  w = softmax(s),  o_h = sum_j w_j V_j.
//
// Work split.  The keys of each (row b, kv head g) are cut into chunks of
// 64 positions; the chunks of all rows, ordered (b, g, chunk), form one list
// of U units.  CTA i of the G-CTA grid takes the contiguous units
// [U i / G, U (i+1) / G), so every CTA streams about the same number of
// bytes whatever the mix of lengths.  A CTA folds the consecutive chunks of
// one (b, g) into a single running (max m, sum l, acc[64]) per query head
// (online softmax) and writes one partial per such segment, at the slot of
// the segment's first chunk.  The last CTA to finish a (b, g) merges its
// segments in chunk order and writes o (f32, and the f16 hi / lo pair the
// following Q8_0 product reads).
//
// Inside a CTA: warp 4 (one elected lane) streams each unit's K and V rows
// (2 x 16 KB, contiguous in the cache) into a ring of shared-memory stages
// with cp.async.bulk, completion counted on an mbarrier per stage; warps 0-3
// consume.  Warp w takes keys 16w .. 16w+15 of the chunk, four at a time:
// lane (k4 = lane / 8, c8 = lane % 8) holds dims 4 c8 .. 4 c8 + 3 and
// 32 + 4 c8 .. 32 + 4 c8 + 3 of key 4t + k4 (two conflict-free 16-byte
// shared loads) and the same dims of every query head in registers; its 8
// partial dot products are reduce-scattered over the 8 lanes of the key
// (xor 4, 2, 1), leaving lane c8 with the score of head c8.
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace qwen2 {
namespace fd {

constexpr int kDh = 64;                 // head dim
constexpr int kCh = 64;                 // keys per unit
constexpr int kStages = 3;
constexpr int kConsumers = 4;           // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kMaxRows = 32;            // rows (sequences) per launch
constexpr int kMaxChunks = 64;          // n_ctx <= 4096
constexpr int kPart = kDh + 2;    // partial: m, l, acc[64]
constexpr unsigned long long kWaitNs = 2000000000ull;

struct Args {
    const float* q;         // [B][nh][64] rotated queries
    const float* kv;        // cache [slots][L][2][nkv][n_ctx][64]
    const int* pos;         // [B] position of each row (attends to 0..pos)
    const int* slot;        // [B] cache slot of each row
    float* part;            // partials [slots... indexed by row b][nh][max_chunks][66]
    int* count;             // [B][nkv] arrival counters, zero between launches
    float* o;               // [B][nh][64]
    __half* o_hi;           // nullable [B][nh][64]
    __half* o_lo;
    int* err;
    int B, nh, nkv, n_ctx, L, layer, max_chunks;
};

struct Smem {
    float ring[kStages][2][kCh][kDh];   // K rows then V rows of one unit
    float wacc[kConsumers][8][kDh];     // per-warp segment accumulators
    float wm[kConsumers][8];
    float wl[kConsumers][8];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int base[kMaxRows + 1];             // first unit of each row
    int nch[kMaxRows];                  // chunks of each row (0 if its position is invalid)
    int posv[kMaxRows];                 // position of each row
    int segs[kMaxChunks];               // merge: first chunk of each segment
    int nseg;
    int last;
    int abort;                          // a bounded wait gave up: skip the remaining work
};

static_assert(sizeof(float) * 2 * 8 * kMaxChunks <= sizeof(float) * kConsumers * 8 * kDh,
              "the merge's per-segment maxima and sums fit in the warp accumulators");

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// First unit of CTA i, and the CTA whose range holds unit u.
__device__ __forceinline__ int unit_start(unsigned i, unsigned U, unsigned G) { return (int)((i * U) / G); }
__device__ __forceinline__ int unit_cta(unsigned u, unsigned U, unsigned G) {
    const unsigned c = ((u + 1) * G - 1) / U;
    return (int)(c < G ? c : G - 1);
}

struct Unit {
    int b, g, c, nj;
};

__device__ __forceinline__ Unit decode_unit(const Smem& sm, int B, int u) {
    int b = 0;
    while (b + 1 < B && sm.base[b + 1] <= u) ++b;
    const int r = u - sm.base[b];
    Unit t;
    t.b = b;
    t.g = r / sm.nch[b];
    t.c = r - t.g * sm.nch[b];
    t.nj = min(kCh, sm.posv[b] + 1 - t.c * kCh);
    return t;
}

__device__ __forceinline__ const float* kv_rows(const Args& a, int b, int which, int g, int p0) {
    const size_t slot = (size_t)a.slot[b];
    return a.kv + ((((slot * a.L + a.layer) * 2 + which) * a.nkv + g) * (size_t)a.n_ctx + p0) * kDh;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            sm100::smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(sm100::smem_addr(bar))
        : "memory");
}

// Is chunk c of (b, g) the first chunk of a segment (of the CTA that holds it)?
__device__ __forceinline__ bool seg_start(const Smem& sm, int b, int g, int c, unsigned U, unsigned G) {
    if (c == 0) return true;
    const unsigned u = (unsigned)(sm.base[b] + g * sm.nch[b] + c);
    return unit_start((unsigned)unit_cta(u, U, G), U, G) == (int)u;
}

// Sum of v[h] over the 8 lanes of a key (lanes differing in bits 0-2),
// scattered so that lane c8 returns head c8's total: halves are exchanged
// over xor 4, then quarters over xor 2, then singles over xor 1.
__device__ __forceinline__ float reduce_scatter8(const float (&v)[8], int c8) {
    const bool b2 = (c8 & 4) != 0, b1 = (c8 & 2) != 0, b0 = (c8 & 1) != 0;
    float w4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b2 ? v[i] : v[i + 4];
        const float keep = b2 ? v[i + 4] : v[i];
        w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float w2[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b1 ? w4[i] : w4[i + 2];
        const float keep = b1 ? w4[i + 2] : w4[i];
        w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    const float send = b0 ? w2[0] : w2[1];
    const float keep = b0 ? w2[1] : w2[0];
    return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

}  // namespace fd

// NG: query-head slots per lane group (7 when the group is exactly 7,
// otherwise 8 with the heads past the group masked).  Grid: any number of
// CTAs (two per SM fit); block fd::kThreads; dynamic shared memory
// sizeof(fd::Smem).
template <int NG>
__global__ void __launch_bounds__(fd::kThreads, 2) k_attn_flash(fd::Args a) {
    using namespace fd;
    extern __shared__ __align__(128) unsigned char fd_smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(fd_smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int group = a.nh / a.nkv;
    if (group > NG || a.B > kMaxRows) {
        if (tid == 0 && blockIdx.x == 0) raise_guard(a.err, kGuardShape);
        return;
    }
    if (warp == 0) {
        // Row table: chunks per row and the first unit of each row.
        int n = 0, p = 0;
        if (lane < a.B) {
            p = a.pos[lane];
            if (p < 0 || p >= a.n_ctx) {
                if (blockIdx.x == 0) raise_guard(a.err, kGuardPosition);
                p = 0;
            } else if ((p + kCh) / kCh > min(a.max_chunks, kMaxChunks)) {
                if (blockIdx.x == 0) raise_guard(a.err, kGuardShape);
                p = 0;
            } else {
                n = (p + kCh) / kCh;
            }
        }
        int v = n * a.nkv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        sm.nch[lane] = n;
        sm.posv[lane] = p;
        sm.base[lane + 1] = v;
        if (lane == 0) {
            sm.base[0] = 0;
            sm.abort = 0;
        }
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            sm100::mbar_init(&sm.full[s], 1);
            sm100::mbar_init(&sm.empty[s], kConsumers);
        }
        sm100::mbar_init_fence();
    }
    if (warp < kConsumers) {
        // Key rows past a unit's length keep whatever an earlier unit left:
        // start from zeros so they are always finite (their weight is 0).
        float4* r = reinterpret_cast<float4*>(&sm.ring[0][0][0][0]);
        constexpr int n4 = kStages * 2 * kCh * kDh / 4;
        for (int i = tid; i < n4; i += kConsumers * 32) r[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    const unsigned U = (unsigned)sm.base[a.B], G = gridDim.x;
    const int u0 = unit_start(blockIdx.x, U, G), u1 = unit_start(blockIdx.x + 1, U, G);

    if (warp == kConsumers) {
        // Producer: one lane issues the K and V bulk copies of each unit.
        if (lane == 0) {
            int k = 0;
            for (int u = u0; u < u1; ++u, ++k) {
                const int s = k % kStages;
                if (k >= kStages &&
                    !sm100::mbar_wait(&sm.empty[s], ((k / kStages) & 1) ^ 1, sm100::global_ns() + kWaitNs)) {
                    raise_guard(a.err, kGuardTimeout);
                    break;
                }
                const Unit t = decode_unit(sm, a.B, u);
                const unsigned bytes = (unsigned)t.nj * kDh * 4;
                sm100::mbar_expect_tx(&sm.full[s], 2 * bytes);
                bulk_g2s(&sm.ring[s][0][0][0], kv_rows(a, t.b, 0, t.g, t.c * kCh), bytes, &sm.full[s]);
                bulk_g2s(&sm.ring[s][1][0][0], kv_rows(a, t.b, 1, t.g, t.c * kCh), bytes, &sm.full[s]);
            }
            // Every copy lands before the CTA exits, even after an abort.
            for (int kk = k > kStages ? k - kStages : 0; kk < k; ++kk)
                sm100::mbar_wait(&sm.full[kk % kStages], (kk / kStages) & 1, sm100::global_ns() + kWaitNs);
        }
        return;
    }


    // ---- consumers: warps 0-3 ---------------------------------------------
    const int k4 = lane >> 3, c8 = lane & 7;
    float qr[NG][8], acc[NG][8];
    float m_run = -INFINITY, l_run = 0.f;
    int c_first = 0;
    int k = 0;
    for (int u = u0; u < u1; ++u, ++k) {
        const Unit t = decode_unit(sm, a.B, u);
        if (u == u0 || t.c == 0) {
            // A new segment: this (b, g)'s query heads, fresh running state.
            c_first = t.c;
            const float* qb = a.q + ((size_t)t.b * a.nh + (size_t)t.g * group) * kDh;
#pragma unroll
            for (int h = 0; h < NG; ++h) {
                float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
                if (h < group) {
                    x0 = *reinterpret_cast<const float4*>(qb + h * kDh + 4 * c8);
                    x1 = *reinterpret_cast<const float4*>(qb + h * kDh + 32 + 4 * c8);
                }
                qr[h][0] = x0.x; qr[h][1] = x0.y; qr[h][2] = x0.z; qr[h][3] = x0.w;
                qr[h][4] = x1.x; qr[h][5] = x1.y; qr[h][6] = x1.z; qr[h][7] = x1.w;
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[h][i] = 0.f;
            }
            m_run = -INFINITY;
            l_run = 0.f;
        }
        const int s = k % kStages;
        bool ok = *reinterpret_cast<volatile int*>(&sm.abort) == 0;
        if (ok && !sm100::mbar_wait(&sm.full[s], (k / kStages) & 1, sm100::global_ns() + kWaitNs)) {
            raise_guard(a.err, kGuardTimeout);
            sm.abort = 1;
            ok = false;
        }
        if (ok) {
            const float* Ks = &sm.ring[s][0][0][0];
            const float* Vs = &sm.ring[s][1][0][0];
            // Scores of keys 16 warp + 4 i + k4 for head c8.
            float sc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 16 * warp + 4 * i + k4;
                const float4 ka = *reinterpret_cast<const float4*>(Ks + j * kDh + 4 * c8);
                const float4 kb = *reinterpret_cast<const float4*>(Ks + j * kDh + 32 + 4 * c8);
                float v[8];
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    if (h < NG) {
                        float d = qr[h][0] * ka.x;
                        d = fmaf(qr[h][1], ka.y, d);
                        d = fmaf(qr[h][2], ka.z, d);
                        d = fmaf(qr[h][3], ka.w, d);
                        d = fmaf(qr[h][4], kb.x, d);
                        d = fmaf(qr[h][5], kb.y, d);
                        d = fmaf(qr[h][6], kb.z, d);
                        d = fmaf(qr[h][7], kb.w, d);
                        v[h] = d;
                    } else {
                        v[h] = 0.f;
                    }
                }
                const float r = reduce_scatter8(v, c8);
                // hd = 64: the scale 1/8 is exact.
                sc[i] = (j < t.nj && c8 < group) ? r * 0.125f : -INFINITY;
            }
            // Online softmax over this warp's 16 keys (per head c8).
            float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
            const float m_new = fmaxf(m_run, mt);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = expf(m_run - m_use);
            float p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = expf(sc[i] - m_use);
            l_run = fmaf(l_run, alpha, (p[0] + p[1]) + (p[2] + p[3]));
            m_run = m_new;
            if (__any_sync(0xffffffffu, c8 < group && alpha != 1.f)) {
#pragma unroll
                for (int h = 0; h < NG; ++h) {
                    const float ah = __shfl_sync(0xffffffffu, alpha, h);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[h][e] *= ah;
                }
            }
            // acc[h] += p[h][j] * V[j] over this lane's keys.
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 16 * warp + 4 * i + k4;
                const float4 va = *reinterpret_cast<const float4*>(Vs + j * kDh + 4 * c8);
                const float4 vb = *reinterpret_cast<const float4*>(Vs + j * kDh + 32 + 4 * c8);
#pragma unroll
                for (int h = 0; h < NG; ++h) {
                    const float ph = __shfl_sync(0xffffffffu, p[i], (k4 << 3) | h);
                    acc[h][0] = fmaf(ph, va.x, acc[h][0]);
                    acc[h][1] = fmaf(ph, va.y, acc[h][1]);
                    acc[h][2] = fmaf(ph, va.z, acc[h][2]);
                    acc[h][3] = fmaf(ph, va.w, acc[h][3]);
                    acc[h][4] = fmaf(ph, vb.x, acc[h][4]);
                    acc[h][5] = fmaf(ph, vb.y, acc[h][5]);
                    acc[h][6] = fmaf(ph, vb.z, acc[h][6]);
                    acc[h][7] = fmaf(ph, vb.w, acc[h][7]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) sm100::mbar_arrive(&sm.empty[s]);

        if (t.c != sm.nch[t.b] - 1 && u + 1 != u1) continue;
        // ---- end of a segment: combine the 4 warps, write one partial ------
        float lt = l_run;
        lt += __shfl_xor_sync(0xffffffffu, lt, 8);
        lt += __shfl_xor_sync(0xffffffffu, lt, 16);
#pragma unroll
        for (int h = 0; h < NG; ++h)
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], 8);
                acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], 16);
            }
        if (k4 == 0) {
#pragma unroll
            for (int h = 0; h < NG; ++h) {
                *reinterpret_cast<float4*>(&sm.wacc[warp][h][4 * c8]) =
                    make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
                *reinterpret_cast<float4*>(&sm.wacc[warp][h][32 + 4 * c8]) =
                    make_float4(acc[h][4], acc[h][5], acc[h][6], acc[h][7]);
            }
            sm.wm[warp][c8] = m_run;
            sm.wl[warp][c8] = lt;
        }
        consumers_sync();
        const size_t head0 = (size_t)t.b * a.nh + (size_t)t.g * group;
        for (int e = tid; e < group * kDh; e += kConsumers * 32) {
            const int h = e >> 6, d = e & 63;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, sm.wm[w][h]);
            float A = 0.f, Lsum = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float wt = sm.wm[w][h] == -INFINITY ? 0.f : expf(sm.wm[w][h] - M);
                A = fmaf(wt, sm.wacc[w][h][d], A);
                Lsum = fmaf(wt, sm.wl[w][h], Lsum);
            }
            float* pr = a.part + ((head0 + h) * a.max_chunks + c_first) * kPart;
            pr[2 + d] = A;
            if (d == 0) {
                pr[0] = M;
                pr[1] = Lsum;
            }
        }
        __threadfence();
        consumers_sync();
        if (warp == 0) {
            // Count this (b, g)'s segments; the CTA that brings the count to
            // that number merges them.
            const int nch = sm.nch[t.b];
            const bool s0 = lane < nch && seg_start(sm, t.b, t.g, lane, U, G);
            const bool s1 = lane + 32 < nch && seg_start(sm, t.b, t.g, lane + 32, U, G);
            const unsigned m0 = __ballot_sync(0xffffffffu, s0), m1 = __ballot_sync(0xffffffffu, s1);
            const int nseg = __popc(m0) + __popc(m1);
            int prev = 0;
            if (lane == 0) prev = atomicAdd(&a.count[t.b * a.nkv + t.g], 1);
            prev = __shfl_sync(0xffffffffu, prev, 0);
            const bool last = prev == nseg - 1;
            if (last) {
                const unsigned lt_mask = (1u << lane) - 1u;
                if (s0) sm.segs[__popc(m0 & lt_mask)] = lane;
                if (s1) sm.segs[__popc(m0) + __popc(m1 & lt_mask)] = lane + 32;
            }
            if (lane == 0) {
                sm.nseg = nseg;
                sm.last = last ? 1 : 0;
            }
        }
        consumers_sync();
        if (sm.last) {
            // Merge the segments in chunk order (all loads of a step issued
            // together): per head M = max m_s, then the weights e^(m_s - M)
            // and L = sum e^(m_s - M) l_s, then o = sum e^(m_s - M) acc_s / L.
            __threadfence();
            const int nseg = sm.nseg;
            float* ms = &sm.wacc[0][0][0];   // [8][kMaxChunks] segment maxima, then weights
            float* ls = ms + 8 * kMaxChunks; // [8][kMaxChunks] segment sums
            for (int e = tid; e < group * nseg; e += kConsumers * 32) {
                const int h = e % group, i = e / group;
                const float* pc = a.part + ((head0 + h) * a.max_chunks + sm.segs[i]) * kPart;
                ms[h * kMaxChunks + i] = __ldcg(pc);
                ls[h * kMaxChunks + i] = __ldcg(pc + 1);
            }
            consumers_sync();
            if (tid < group) {
                const int h = tid;
                float M = -INFINITY;
                for (int i = 0; i < nseg; ++i) M = fmaxf(M, ms[h * kMaxChunks + i]);
                float Lsum = 0.f;
                for (int i = 0; i < nseg; ++i) {
                    const float wt = expf(ms[h * kMaxChunks + i] - M);
                    ms[h * kMaxChunks + i] = wt;
                    Lsum = fmaf(wt, ls[h * kMaxChunks + i], Lsum);
                }
                sm.wl[0][h] = Lsum;
            }
            consumers_sync();
            for (int e = tid; e < group * kDh; e += kConsumers * 32) {
                const int h = e >> 6, d = e & 63;
                const float* ph = a.part + (head0 + h) * a.max_chunks * kPart + 2 + d;
                float O = 0.f;
                for (int i0 = 0; i0 < nseg; i0 += 8) {
                    float v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        v[j] = i0 + j < nseg ? __ldcg(ph + sm.segs[i0 + j] * kPart) : 0.f;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (i0 + j < nseg) O = fmaf(ms[h * kMaxChunks + i0 + j], v[j], O);
                }
                const float ov = O / sm.wl[0][h];
                const size_t oi = (head0 + h) * kDh + d;
                a.o[oi] = ov;
                if (a.o_hi) {
                    const __half hi = __float2half_rn(ov);
                    a.o_hi[oi] = hi;
                    a.o_lo[oi] = __float2half_rn(ov - __half2float(hi));
                }
            }
            if (tid == 0) a.count[t.b * a.nkv + t.g] = 0;
        }
        consumers_sync();
    }
}

}  // namespace qwen2
