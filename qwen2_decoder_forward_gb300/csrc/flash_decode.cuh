// Batched GQA decode attention over an f32 KV cache, for many sequences at
// ragged positions in one launch (flash-decoding with a persistent grid and
// warp-level TF32 tensor-core products).
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
// the segment's first chunk.  k_attn_merge, launched next, merges the
// segments of each (b, g) in chunk order and writes o (f32, and the f16
// hi / lo pair the following Q8_0 product reads).
//
// Inside a CTA: warp 4 (one elected lane) loads each unit's K and V tiles
// (64 positions x 64 floats each) with four TMA tensor copies into a ring
// of shared-memory stages (128-byte swizzle, so the fragment loads below
// are conflict-free), completion counted on an mbarrier per stage; warps
// 0-3 consume, warp w taking keys 16w .. 16w + 15 of the chunk:
//   scores  S^T[key][head] = K[key][:] . Q[head][:]   (m16n8k8, M = 16 keys,
//           N = 8 head slots, K = 8 dims per step, 8 steps);
//   values  O^T[dim][head] += V^T[dim][key] . P^T[key][head] (M = 16 dims,
//           4 tiles, K = 8 keys per step, 2 steps).
// Precision: q, k and the probabilities enter the MMAs rounded to TF32
// (10-bit mantissa, round to nearest); v enters as a TF32 hi / lo pair (two
// MMAs), the same split the tensor-core prefill uses for v; the softmax
// statistics, the sums l (of the rounded probabilities) and the accumulators
// are f32.  The softmax runs in base 2 (scores scaled by log2(e) / 8,
// exponentials by ex2); a partial's maximum is stored in natural-log units.
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace qwen2 {
namespace fd {

constexpr int kDh = 64;                 // head dim
constexpr int kCh = 64;                 // keys per unit
constexpr int kStages = 2;
constexpr int kConsumers = 4;           // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kMaxRows = 32;            // rows (sequences) per launch
constexpr int kMaxChunks = 64;          // n_ctx <= 4096
constexpr int kGroupMax = 8;            // query heads per kv head
constexpr int kPart = kDh + 2;          // partial: m, l, acc[64]
constexpr int kHalf = kCh * 32;         // floats of one swizzled half tile (64 rows x 128 bytes)
constexpr unsigned kUnitBytes = 4u * kHalf * 4u;  // K and V, two halves each

struct Args {
    const float* q;         // [B][nh][64] rotated queries
    const int* pos;         // [B] position of each row (attends to 0..pos)
    const int* slot;        // [B] cache slot of each row
    float* part;            // partials [B][nh][max_chunks][66]
    int* count;             // [B][nkv] arrival counters, zero between launches
    float* o;               // [B][nh][64]
    __half* o_hi;           // nullable [B][nh][64]
    __half* o_lo;
    int* err;
    int B, nh, nkv, n_ctx, L, layer, max_chunks;
    const unsigned char* pf;  // nullable: bytes to prefetch into L2 for the kernels that follow
    size_t pf_bytes;          // (a multiple of 16, 16-byte aligned)
};

struct Smem {
    // [stage][K, V][dims 0-31, 32-63][row][32 floats], each half tile
    // 128-byte swizzled (1024-byte aligned).
    float ring[kStages][2][2][kHalf];
    float qs[kStages][kGroupMax * kDh];    // the unit's query heads, when it starts a segment
    float wacc[kConsumers][kGroupMax][kDh];  // per-warp segment accumulators
    float wm[kConsumers][kGroupMax];
    float wl[kConsumers][kGroupMax];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int base[kMaxRows + 1];             // first unit of each row
    int nch[kMaxRows];                  // chunks of each row (0 if its position is invalid)
    int posv[kMaxRows];                 // position of each row
    int slotv[kMaxRows];                // cache slot of each row
    int abort;                          // a bounded wait gave up: skip the remaining work
};
// Dynamic shared memory to request: the ring needs 1024-byte alignment.
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;


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

// The unit after t in (b, g, c) order (rows without chunks skipped); only
// called while a next unit exists.
__device__ __forceinline__ void next_unit(const Smem& sm, int B, int nkv, Unit& t) {
    if (++t.c >= sm.nch[t.b]) {
        t.c = 0;
        if (++t.g >= nkv) {
            t.g = 0;
            do {
                ++t.b;
            } while (t.b + 1 < B && sm.nch[t.b] == 0);
        }
    }
    t.nj = min(kCh, sm.posv[t.b] + 1 - t.c * kCh);
}

// 2^x by the MUFU instruction (relative error about 2^-22; the
// probabilities are rounded to TF32 afterwards).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// Row of the cache viewed as a [rows][64] f32 matrix: position p0 of
// (slot, layer, K or V, kv head g).
__device__ __forceinline__ int kv_row(const Args& a, int slot, int which, int g, int p0) {
    return (((slot * a.L + a.layer) * 2 + which) * a.nkv + g) * a.n_ctx + p0;
}

// Is chunk c of (b, g) the first chunk of a segment (of the CTA that holds it)?
__device__ __forceinline__ bool seg_start(const int* base, const int* nch, int b, int g, int c, unsigned U,
                                          unsigned G) {
    if (c == 0) return true;
    const unsigned u = (unsigned)(base[b] + g * nch[b] + c);
    return unit_start((unsigned)unit_cta(u, U, G), U, G) == (int)u;
}

// Float index of element (row, f) (f < 32) in a 128-byte-swizzled half tile:
// the 16-byte chunk f / 4 of row r sits at chunk (f / 4) ^ (r % 8).
__device__ __forceinline__ int swz(int row, int f) { return row * 32 + ((((f >> 2) ^ (row & 7)) << 2) | (f & 3)); }

// Four 8 x 8 matrices of 16-bit elements from shared memory (each lane
// gives one 16-byte row address); for 32-bit data each matrix is 8 rows x 4
// words and thread i receives word i % 4 of row i / 4.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const float* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"((uint32_t)__cvta_generic_to_shared(p)));
}

__device__ __forceinline__ uint32_t tf32_rn(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

using sm100::bulk_g2s;

// Row table of a launch (warp 0 of the block): per row its position, slot
// and chunk count (0 if the position is invalid) and its first unit.
__device__ __forceinline__ void row_table(const Args& a, int* base, int* nch, int* posv, int* slotv) {
    const int lane = threadIdx.x & 31;
    int n = 0, p = 0, sl = 0;
    if (lane < a.B) {
        p = a.pos[lane];
        sl = a.slot[lane];
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
    nch[lane] = n;
    if (posv) posv[lane] = p;
    if (slotv) slotv[lane] = sl;
    base[lane + 1] = v;
    if (lane == 0) base[0] = 0;
}

// d += a . b for one 16 x 8 x 8 TF32 tile (f32 accumulation).
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

}  // namespace fd
}  // namespace qwen2

namespace qwen2 {

// Grid: any number of CTAs (two per SM fit); block fd::kThreads; dynamic
// shared memory fd::kSmemBytes.  kvmap: the KV cache as a [rows][64] f32
// matrix (rows = slots * L * 2 * nkv * n_ctx), boxes of 32 floats x 64 rows,
// 128-byte swizzle.
__global__ void __launch_bounds__(fd::kThreads, 2)
    k_attn_flash(const __grid_constant__ CUtensorMap kvmap, fd::Args a) {
    using namespace fd;
    extern __shared__ unsigned char fd_smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(fd_smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int group = a.nh / a.nkv;
    if (group > kGroupMax || a.B > kMaxRows) {
        if (tid == 0 && blockIdx.x == 0) raise_guard(a.err, kGuardShape);
        return;
    }
    pdl_launch_dependents();
    // Positions and slots are written only by the LM head at the end of the
    // previous step, which has completed before this step's first kernel
    // (launched without the PDL attribute) starts: the row table can be
    // built while the previous kernel drains.
    if (warp == 0) {
        row_table(a, sm.base, sm.nch, sm.posv, sm.slotv);
        if (lane == 0) sm.abort = 0;
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            sm100::mbar_init(&sm.full[s], 1);
            sm100::mbar_init(&sm.empty[s], kConsumers);
        }
        sm100::mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();  // q and the new keys come from the previous kernel
    const unsigned U = (unsigned)sm.base[a.B], G = gridDim.x;
    const int u0 = unit_start(blockIdx.x, U, G), u1 = unit_start(blockIdx.x + 1, U, G);

    if (warp == kConsumers) {
        // Producer: one lane issues the four tensor copies of each unit.
        if (lane == 0) {
            sm100::tma_prefetch_desc(&kvmap);
            // This CTA's share of the weights the next products stream: the
            // attention leaves DRAM bandwidth over, so they can wait in L2.
            if (a.pf) {
                const size_t share = (a.pf_bytes / gridDim.x + 15) & ~(size_t)15;
                const size_t b0 = share * blockIdx.x;
                const size_t b1 = min(a.pf_bytes, b0 + share);
                for (size_t o = b0; o < b1; o += 16384)
                    sm100::prefetch_l2(a.pf + o, (unsigned)min((size_t)16384, b1 - o));
            }
            // K and V are read once: first out of L2.
            const uint64_t pol = sm100::policy_evict_first();
            int k = 0;
            Unit t{};
            if (u0 < u1) t = decode_unit(sm, a.B, u0);
            for (int u = u0; u < u1; ++u, ++k) {
                const int s = k % kStages;
                if (k >= kStages &&
                    !sm100::mbar_wait(&sm.empty[s], ((k / kStages) & 1) ^ 1, kWaitNs)) {
                    raise_guard(a.err, kGuardTimeout);
                    break;
                }
                if (u != u0) next_unit(sm, a.B, a.nkv, t);
                const int yk = kv_row(a, sm.slotv[t.b], 0, t.g, t.c * kCh);
                const int yv = kv_row(a, sm.slotv[t.b], 1, t.g, t.c * kCh);
                // A unit that starts a segment also brings its query heads.
                const bool first = u == u0 || t.c == 0;
                const unsigned qbytes = first ? (unsigned)(group * kDh * 4) : 0u;
                sm100::mbar_expect_tx(&sm.full[s], kUnitBytes + qbytes);
                if (first)
                    bulk_g2s(sm.qs[s], a.q + ((size_t)t.b * a.nh + (size_t)t.g * group) * kDh, qbytes, &sm.full[s]);
                sm100::tma_load_2d_hint(sm.ring[s][0][0], &kvmap, 0, yk, &sm.full[s], pol);
                sm100::tma_load_2d_hint(sm.ring[s][0][1], &kvmap, 32, yk, &sm.full[s], pol);
                sm100::tma_load_2d_hint(sm.ring[s][1][0], &kvmap, 0, yv, &sm.full[s], pol);
                sm100::tma_load_2d_hint(sm.ring[s][1][1], &kvmap, 32, yv, &sm.full[s], pol);
            }
            // Every copy lands before the CTA exits, even after an abort.
            for (int kk = k > kStages ? k - kStages : 0; kk < k; ++kk)
                sm100::mbar_wait(&sm.full[kk % kStages], (kk / kStages) & 1, kWaitNs);
        }
        return;
    }

    // ---- consumers: warps 0-3 ---------------------------------------------
    const int g8 = lane >> 2, t4 = lane & 3;   // fragment row group, thread in group
    const int key0 = 16 * warp;                // this warp's keys within a chunk
    const int h0 = 2 * t4, h1 = 2 * t4 + 1;    // the two head slots of this thread's scores / outputs
    uint32_t qb[8][2];                         // B fragments of Q^T (TF32), per 8-dim step
    float oacc[4][4];                          // O^T[16 mt + g8 (+8)][h0, h1]
    float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;
    int c_first = 0;
    int k = 0;
    Unit t{};
    if (u0 < u1) t = decode_unit(sm, a.B, u0);
    for (int u = u0; u < u1; ++u, ++k) {
        if (u != u0) next_unit(sm, a.B, a.nkv, t);
        const int s = k % kStages;
        bool ok = *reinterpret_cast<volatile int*>(&sm.abort) == 0;
        if (ok && !sm100::mbar_wait(&sm.full[s], (k / kStages) & 1, kWaitNs)) {
            raise_guard(a.err, kGuardTimeout);
            sm.abort = 1;
            ok = false;
        }
        if (u == u0 || t.c == 0) {
            // A new segment: this (b, g)'s query heads (brought with the
            // unit), fresh running state.
            c_first = t.c;
            const float* qh = sm.qs[s] + g8 * kDh;
#pragma unroll
            for (int s8 = 0; s8 < 8; ++s8) {
                const bool hv = ok && g8 < group;
                qb[s8][0] = tf32_rn(hv ? qh[8 * s8 + t4] : 0.f);
                qb[s8][1] = tf32_rn(hv ? qh[8 * s8 + t4 + 4] : 0.f);
            }
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
            m_run0 = m_run1 = -INFINITY;
            l_run0 = l_run1 = 0.f;
        }
        if (ok) {
            const float* Kt = sm.ring[s][0][0];
            const float* Vt = sm.ring[s][1][0];
            // Scores S^T[key0 + g8 (+8)][h0, h1] over the 64 dims, as two
            // independent chains (dims 0-31, 32-63) added at the end.
            // The A fragment of each 8-dim step in one ldmatrix.x4: matrix
            // j (lanes 8j .. 8j + 7 give its row addresses) is keys key0 +
            // 8 (j & 1) + 0..7 by the 4 dims (16 bytes) 4 (j >> 1) .. + 3 of
            // the step, so thread (g8, t4) receives K[key0 + g8 (+8)][dim
            // t4 (+4)] as fragments a0..a3.
            float sc[4] = {0.f, 0.f, 0.f, 0.f}, sc2[4] = {0.f, 0.f, 0.f, 0.f};
            const int lrow = key0 + (lane & 7) + 8 * ((lane >> 3) & 1);
            const int lchunk = lane >> 4;  // 0: dims 0-3 of the step, 1: dims 4-7
#pragma unroll
            for (int s8 = 0; s8 < 8; ++s8) {
                const float* Kh = Kt + (s8 >> 2) * kHalf;
                const int c = 2 * (s8 & 3) + lchunk;  // 16-byte chunk of the row's 128 bytes
                uint32_t r[4];
                ldsm_x4(r, Kh + lrow * 32 + ((c ^ (lrow & 7)) << 2));
                uint32_t af[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) af[i] = tf32_rn(__uint_as_float(r[i]));
                if (s8 < 4) mma_tf32(sc, af, qb[s8][0], qb[s8][1]);
                else mma_tf32(sc2, af, qb[s8][0], qb[s8][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[i] += sc2[i];
            // hd = 64: the scale 1/8 is exact.  Keys past the chunk's length
            // and head slots past the group get -inf.
            const bool klo = key0 + g8 < t.nj, khi = key0 + g8 + 8 < t.nj;
            const bool v0 = h0 < group, v1 = h1 < group;
            // Scores in base-2 units (log2 e folded into the 1/8): the
            // running maxima and the exponentials below use 2^x.
            constexpr float kS2 = 0.125f * kLog2e;
            sc[0] = (klo && v0) ? sc[0] * kS2 : -INFINITY;
            sc[1] = (klo && v1) ? sc[1] * kS2 : -INFINITY;
            sc[2] = (khi && v0) ? sc[2] * kS2 : -INFINITY;
            sc[3] = (khi && v1) ? sc[3] * kS2 : -INFINITY;
            // Online softmax over this warp's 16 keys, per head slot.
            float mt0 = fmaxf(sc[0], sc[2]), mt1 = fmaxf(sc[1], sc[3]);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, o));
                mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, o));
            }
            const float mn0 = fmaxf(m_run0, mt0), mn1 = fmaxf(m_run1, mt1);
            const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = ex2(m_run0 - mu0), al1 = ex2(m_run1 - mu1);
            m_run0 = mn0;
            m_run1 = mn1;
            // Probabilities rounded to TF32 here, so l sums what the MMA uses.
            uint32_t pb[4];
            pb[0] = tf32_rn(ex2(sc[0] - mu0));
            pb[1] = tf32_rn(ex2(sc[1] - mu1));
            pb[2] = tf32_rn(ex2(sc[2] - mu0));
            pb[3] = tf32_rn(ex2(sc[3] - mu1));
            l_run0 = fmaf(l_run0, al0, __uint_as_float(pb[0]) + __uint_as_float(pb[2]));
            l_run1 = fmaf(l_run1, al1, __uint_as_float(pb[1]) + __uint_as_float(pb[3]));
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                oacc[mt][0] *= al0;
                oacc[mt][1] *= al1;
                oacc[mt][2] *= al0;
                oacc[mt][3] *= al1;
            }
            // O^T += V^T . P^T.  Within each 8-key step the k index runs
            // over keys in the order 0, 2, 4, 6 (k = 0..3) and 1, 3, 5, 7
            // (k = 4..7), so thread (g8, t4) needs P[key 2 t4 (+1)][head g8]:
            // scores of key j sit in thread (j % 8, head / 2) as component
            // (head % 2) + 2 (j / 8).
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int src0 = (2 * t4) * 4 + (g8 >> 1), src1 = (2 * t4 + 1) * 4 + (g8 >> 1);
                const uint32_t e0 = __shfl_sync(0xffffffffu, pb[2 * kk], src0);
                const uint32_t o0 = __shfl_sync(0xffffffffu, pb[2 * kk + 1], src0);
                const uint32_t e1 = __shfl_sync(0xffffffffu, pb[2 * kk], src1);
                const uint32_t o1 = __shfl_sync(0xffffffffu, pb[2 * kk + 1], src1);
                const uint32_t b0 = (g8 & 1) ? o0 : e0, b1 = (g8 & 1) ? o1 : e1;
                const int r0 = key0 + 8 * kk + 2 * t4;  // keys of k = t4 and k = t4 + 4
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    const float* Vh = Vt + (mt >> 1) * kHalf;
                    const int f = 16 * (mt & 1) + g8;
                    const float va = Vh[swz(r0, f)], vb = Vh[swz(r0, f + 8)];
                    const float vc = Vh[swz(r0 + 1, f)], vd = Vh[swz(r0 + 1, f + 8)];
                    uint32_t ah[4], alo[4];
                    ah[0] = tf32_rn(va);
                    ah[1] = tf32_rn(vb);
                    ah[2] = tf32_rn(vc);
                    ah[3] = tf32_rn(vd);
                    alo[0] = __float_as_uint(va - __uint_as_float(ah[0]));
                    alo[1] = __float_as_uint(vb - __uint_as_float(ah[1]));
                    alo[2] = __float_as_uint(vc - __uint_as_float(ah[2]));
                    alo[3] = __float_as_uint(vd - __uint_as_float(ah[3]));
                    mma_tf32(oacc[mt], ah, b0, b1);
                    mma_tf32(oacc[mt], alo, b0, b1);
                }
            }
        }
        __syncwarp();
        if (lane == 0) sm100::mbar_arrive(&sm.empty[s]);

        if (t.c != sm.nch[t.b] - 1 && u + 1 != u1) continue;
        // ---- end of a segment: combine the 4 warps, write one partial ------
        float lt0 = l_run0, lt1 = l_run1;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
            lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
        }
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const int d = 16 * mt + g8;
            sm.wacc[warp][h0][d] = oacc[mt][0];
            sm.wacc[warp][h1][d] = oacc[mt][1];
            sm.wacc[warp][h0][d + 8] = oacc[mt][2];
            sm.wacc[warp][h1][d + 8] = oacc[mt][3];
        }
        if (g8 == 0) {
            sm.wm[warp][h0] = m_run0;
            sm.wm[warp][h1] = m_run1;
            sm.wl[warp][h0] = lt0;
            sm.wl[warp][h1] = lt1;
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
                const float wt = sm.wm[w][h] == -INFINITY ? 0.f : ex2(sm.wm[w][h] - M);
                A = fmaf(wt, sm.wacc[w][h][d], A);
                Lsum = fmaf(wt, sm.wl[w][h], Lsum);
            }
            float* pr = a.part + ((head0 + h) * a.max_chunks + c_first) * kPart;
            pr[2 + d] = A;
            if (d == 0) {
                pr[0] = M / kLog2e;  // the partial's maximum in natural-log units, as the merge reads it
                pr[1] = Lsum;
            }
        }
        consumers_sync();
    }
}

// Merge of the segments k_attn_flash wrote for one (row b, kv head g) per
// block (grid B * nkv, kMergeThreads threads; thread e takes output (head
// e / 64, dim e % 64)), in chunk order: M = max m_s, L = sum e^(m_s - M)
// l_s, o = sum e^(m_s - M) acc_s / L (f32, and the f16 hi / lo pair when
// o_hi is set).  Each thread issues the loads of eight segments at once.
// flash_grid: the grid size the attention ran with (it fixes the segments).
constexpr int kMergeThreads = fd::kGroupMax * fd::kDh;
__global__ void __launch_bounds__(kMergeThreads) k_attn_merge(fd::Args a, int flash_grid) {
    using namespace fd;
    __shared__ int base[kMaxRows + 1], nch[kMaxRows], segs[kMaxChunks];
    __shared__ int nseg_s;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int group = a.nh / a.nkv;
    const int b = blockIdx.x / a.nkv, g = blockIdx.x % a.nkv;
    if (group > kGroupMax || a.B > kMaxRows || b >= a.B) return;
    pdl_launch_dependents();
    // The row table and segment list depend on positions only (final for
    // the step, as in k_attn_flash): built before the wait.
    if (warp == 0) {
        row_table(a, base, nch, nullptr, nullptr);
        __syncwarp();
        const unsigned U = (unsigned)base[a.B], G = (unsigned)flash_grid;
        const int n = nch[b];
        const bool s0 = lane < n && seg_start(base, nch, b, g, lane, U, G);
        const bool s1 = lane + 32 < n && seg_start(base, nch, b, g, lane + 32, U, G);
        const unsigned m0 = __ballot_sync(0xffffffffu, s0), m1 = __ballot_sync(0xffffffffu, s1);
        const unsigned lt_mask = (1u << lane) - 1u;
        if (s0) segs[__popc(m0 & lt_mask)] = lane;
        if (s1) segs[__popc(m0) + __popc(m1 & lt_mask)] = lane + 32;
        if (lane == 0) nseg_s = __popc(m0) + __popc(m1);
    }
    __syncthreads();
    pdl_wait();  // the attention's partials
    const int nseg = nseg_s;
    const int h = tid >> 6, d = tid & 63;
    if (nseg == 0 || h >= group) return;  // invalid position: reported by the attention
    const size_t head = (size_t)b * a.nh + (size_t)g * group + h;
    const float* ph = a.part + head * a.max_chunks * kPart;
    float M = -INFINITY, Lsum = 0.f, O = 0.f;
    for (int i0 = 0; i0 < nseg; i0 += 8) {
        float mv[8], lv[8], av[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const bool in = i0 + j < nseg;
            const float* pc = ph + (in ? segs[i0 + j] : 0) * kPart;
            mv[j] = in ? __ldcg(pc) : -INFINITY;
            lv[j] = in ? __ldcg(pc + 1) : 0.f;
            av[j] = in ? __ldcg(pc + 2 + d) : 0.f;
        }
        // Running rescale over groups of eight segments; with nseg <= 8 (the
        // usual case) this is the plain formula.
        float m8 = mv[0];
#pragma unroll
        for (int j = 1; j < 8; ++j) m8 = fmaxf(m8, mv[j]);
        const float Mn = fmaxf(M, m8);
        const float c = M == -INFINITY ? 0.f : expf(M - Mn);
        Lsum *= c;
        O *= c;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float wt = mv[j] == -INFINITY ? 0.f : expf(mv[j] - Mn);
            Lsum = fmaf(wt, lv[j], Lsum);
            O = fmaf(wt, av[j], O);
        }
        M = Mn;
    }
    const float ov = O / Lsum;
    const size_t oi = head * kDh + d;
    a.o[oi] = ov;
    if (a.o_hi) {
        const __half hi = __float2half_rn(ov);
        a.o_hi[oi] = hi;
        a.o_lo[oi] = __float2half_rn(ov - __half2float(hi));
    }
}

}  // namespace qwen2
