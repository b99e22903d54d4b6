// Decode attention arithmetic shared by the per-step attention kernel and the
// persistent decode kernel, so both produce the same bits.
//
// GQA (nnterp encyclopedia qwen2, "Grouped-query attention"): kv head g
// serves query heads g*group .. g*group + group - 1; scores are
// q . k / sqrt(64) over keys 0..p (full causal, no window).  Keys are taken
// in chunks of 64 positions; each chunk yields, per query head, the running
// maximum m, the sum l of e^(s - m) and acc[d] = sum e^(s - m) v[d]; chunks
// are merged in chunk order.
#pragma once

#include "common.cuh"

namespace qwen2 {

constexpr int kHd = 64;        // head_dim of the persistent decode kernel (Qwen2.5-0.5B)
constexpr int kAttCh = 64;     // keys per chunk
constexpr int kMaxGroup = 8;   // query heads per kv head
constexpr int kPartStride = kHd + 2;  // one partial: m, l, acc[64]

// Attention scratch for head_dim HD: q of the group's heads, one chunk of
// keys and values, the chunk's probabilities and softmax statistics.
template <int HD>
struct AttnSmemT {
    float q[kMaxGroup][HD];
    float k[kAttCh][HD + 1];   // padded: lanes read different keys
    float v[kAttCh][HD];
    float p[kMaxGroup][kAttCh];
    float m[kMaxGroup];
    float l[kMaxGroup];
};
using AttnSmem = AttnSmemT<kHd>;

// 1 / sqrt(head_dim): 0.125 exactly for 64, the float nearest 1/sqrt(128)
// for 128.
template <int HD>
__host__ __device__ constexpr float attn_scale() {
    static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
    return HD == 64 ? 0.125f : 0.08838834764831843f;
}

// One chunk of nj <= 64 keys (k, v, q already in `sm`) for `group` query
// heads, computed by a 256-thread group; emit(h, d, acc, m, l) once per
// output element.
template <class S, int HD, class Emit>
__device__ __forceinline__ void attn_chunk(AttnSmemT<HD>& sm, int group, int nj, Emit emit) {
    const int tid = threadIdx.x;
    // Scores q_h . k_j / sqrt(hd); hd = 64 makes the scale 0.125 exact,
    // hd = 128 takes the float nearest 1/sqrt(128).
    for (int e = tid; e < group * kAttCh; e += 256) {
        const int h = e / kAttCh, j = e % kAttCh;
        float s = -INFINITY;
        if (j < nj) {
            // Four partial sums over d = 4i + {0,1,2,3}, added in a fixed order.
            float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
            for (int d = 0; d < HD; d += 4) {
                a0 = fmaf(sm.q[h][d], sm.k[j][d], a0);
                a1 = fmaf(sm.q[h][d + 1], sm.k[j][d + 1], a1);
                a2 = fmaf(sm.q[h][d + 2], sm.k[j][d + 2], a2);
                a3 = fmaf(sm.q[h][d + 3], sm.k[j][d + 3], a3);
            }
            s = ((a0 + a1) + (a2 + a3)) * attn_scale<HD>();
        }
        sm.p[h][j] = s;
    }
    S::sync();
    // Per head (one warp each): max, exponentials, sum.
    const int warp = tid >> 5, lane = tid & 31;
    for (int h = warp; h < group; h += 8) {
        const float s0 = sm.p[h][lane], s1 = sm.p[h][lane + 32];
        const float m = warp_max(fmaxf(s0, s1));
        const float e0 = expf(s0 - m), e1 = expf(s1 - m);
        sm.p[h][lane] = e0;
        sm.p[h][lane + 32] = e1;
        const float l = warp_sum(e0 + e1);
        if (lane == 0) {
            sm.m[h] = m;
            sm.l[h] = l;
        }
    }
    S::sync();
    for (int e = tid; e < group * HD; e += 256) {
        const int h = e / HD, d = e % HD;
        // Four partial sums over keys j = 4i + {0,1,2,3} below nj & ~3, the
        // last nj % 4 keys into the first, then added in a fixed order (rows
        // of v past nj are never read).
        const int nj4 = nj & ~3;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        for (int j = 0; j < nj4; j += 4) {
            a0 = fmaf(sm.p[h][j], sm.v[j][d], a0);
            a1 = fmaf(sm.p[h][j + 1], sm.v[j + 1][d], a1);
            a2 = fmaf(sm.p[h][j + 2], sm.v[j + 2][d], a2);
            a3 = fmaf(sm.p[h][j + 3], sm.v[j + 3][d], a3);
        }
        for (int j = nj4; j < nj; ++j) a0 = fmaf(sm.p[h][j], sm.v[j][d], a0);
        emit(h, d, (a0 + a1) + (a2 + a3), sm.m[h], sm.l[h]);
    }
}

// Merge of n chunk partials for element d of one head:
// M = max m_c, L = sum e^(m_c - M) l_c, o = sum e^(m_c - M) acc_c[d] / L.
// get(c, i) returns field i of chunk c's partial (0: m, 1: l, 2 + d: acc).
template <class Get>
__device__ __forceinline__ float attn_merge(int n, int d, Get get) {
    float M = -INFINITY;
    for (int c = 0; c < n; ++c) M = fmaxf(M, get(c, 0));
    float L = 0.f, O = 0.f;
    for (int c = 0; c < n; ++c) {
        const float w = expf(get(c, 0) - M);
        L = fmaf(w, get(c, 1), L);
        O = fmaf(w, get(c, 2 + d), O);
    }
    return O / L;
}

}  // namespace qwen2
