// Causal GQA attention of the tensor-core prefill (QWEN2_PREFILL_TENSOR) on
// the 5th-generation tensor cores: tcgen05 MMAs from shared memory into
// tensor memory (nnterp encyclopedia qwen2, "Grouped-query attention": kv
// head g serves query heads g*group .. g*group + group - 1; scores
// q . k / sqrt(64) over keys 0..p).
//
// Two kernels per layer; the first (k_att_operands) only when keys stored
// by an earlier call must be brought in.
//
// The attention reads its keys from f16 operand buffers laid out for TMA:
// k as rows [slot][kv head][position][64 dims] and v transposed as an f16
// hi / lo pair, rows [slot][kv head][hi, lo][dim][positions].  The QKV
// product's epilogue writes the call's own rows there as it stores them in
// the f32 cache; k_att_operands converts, from the cache, the positions an
// earlier call stored (those below the sequence's seq_conv).  Positions past
// a sequence's last key inside its last 64-key tile hold stale finite
// values or the buffers' initial zeros: their scores are masked and their
// probabilities are exactly 0.
//
// k_attn_prefill_tc: block (g, blk) takes up to 16 query positions of one
// sequence; their group query heads form the rows of one 128-row tile (row
// r = position r / group, head r % group; rows past 16 * group are padding).
// Per 64-key tile t:
//   S[128 x 64]   = Q[128 x 64] . K_t^T      tcgen05.mma into tensor memory
//   P             = exp(S / 8 - m)           online softmax in registers
//   O_t[128 x 64] = P . (V_t,hi + V_t,lo)    tcgen05.mma into tensor memory
//   O             = O * correction + O_t     in registers, one tile later
// K and V^T tiles arrive by TMA into a three-stage ring (128-byte swizzle,
// the K-major operand layout), two tiles ahead of the products.  One lane
// of warp 4 allocates tensor memory and issues the copies and the MMAs;
// right after each tile's probabilities are in shared memory it issues the
// next tile's scores and this tile's value product (into one of two TMEM
// buffers), so the tensor cores work while the threads fold the previous
// tile's product into their registers.
// Thread (w, lane) owns row 32 (w mod 4) + lane (its TMEM lane), half of
// the score columns and output dims 32 (w / 4) .. + 31; the two threads of
// a row share the row maximum and their partial sums through shared memory.
//
// Precision: q, k and the probabilities enter the MMAs as f16, v as an f16
// hi / lo pair (two MMAs); accumulation, softmax statistics and the output
// are f32, and the output is written as the f16 hi / lo pair o_proj reads.
//
// Every wait is bounded by the global timer; a wait that runs out sets the
// guard word, the block stops at its next check and lets its copies land
// before it returns.
#include "common.cuh"
#include "prefill.h"
#include "sm100.cuh"

namespace qwen2 {

namespace {

constexpr int kThreads = 256;
constexpr int kD = 64;       // head_dim
constexpr int kKT = 64;      // keys per tile
constexpr int kRows = 128;   // MMA M: query rows (positions x heads) per block
constexpr int kStages = 3;   // K / V^T ring
constexpr unsigned kTileBytes = kKT * 128;  // one 64 x 64 f16 operand tile
constexpr uint32_t kTmemCols = 256;         // S, and two value-product buffers
constexpr float kScaleLog2 = 0.125f * 1.4426950408889634f;  // 1/sqrt(64) * log2(e)

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    __half2 h;
    h = __floats2half2_rn(f[0], f[1]); u.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(f[2], f[3]); u.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(f[4], f[5]); u.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2half2_rn(f[6], f[7]); u.w = *reinterpret_cast<uint32_t*>(&h);
    return u;
}

// ---- operand conversion ----------------------------------------------------------

struct OperandArgs {
    const float* kv;
    const int* seq_slot;
    const int* seq_conv;
    __half* att_k;
    __half* att_vt;
    int nkv, n_ctx, n_ctx64, L, layer;
};

// Grid (tiles, sequences, kv heads), 256 threads: the positions below
// seq_conv of one 64-key tile each.
__global__ void __launch_bounds__(256) k_att_operands(OperandArgs a) {
    __shared__ float vs[kKT][kD + 1];
    const int t = blockIdx.x, s = blockIdx.y, g = blockIdx.z, tid = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait();
    const int end = a.seq_conv[s], j0 = t * kKT;
    if (j0 >= end) return;
    const int pmax = end - 1;
    const int slot = a.seq_slot[s];
    const size_t head_stride = (size_t)a.n_ctx * kD;
    const size_t cache0 = ((size_t)slot * a.L + a.layer) * 2 * a.nkv;
    const float* kb = a.kv + (cache0 + g) * head_stride;
    const float* vb = a.kv + (cache0 + a.nkv + g) * head_stride;
    const size_t head = (size_t)slot * a.nkv + g;
    // Every load of the tile is issued before the first use: K as key j,
    // dims c0 .. c0 + 15 per thread; V as four (key, 4-dim) pieces.
    const int j = tid >> 2, c0 = 16 * (tid & 3);
    const bool kin = j0 + j <= pmax;
    float4 kx[4], vx[4];
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4* ksrc = reinterpret_cast<const float4*>(kb + (size_t)(j0 + j) * kD + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i) kx[i] = kin ? ksrc[i] : zero;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = tid + 256 * i, jv = e >> 4, d4 = 4 * (e & 15);
        vx[i] = j0 + jv <= pmax ? *reinterpret_cast<const float4*>(vb + (size_t)(j0 + jv) * kD + d4) : zero;
    }
    if (kin) {
        const float f0[8] = {kx[0].x, kx[0].y, kx[0].z, kx[0].w, kx[1].x, kx[1].y, kx[1].z, kx[1].w};
        const float f1[8] = {kx[2].x, kx[2].y, kx[2].z, kx[2].w, kx[3].x, kx[3].y, kx[3].z, kx[3].w};
        uint4* dst = reinterpret_cast<uint4*>(a.att_k + (head * a.n_ctx64 + j0 + j) * kD + c0);
        dst[0] = pack8(f0);
        dst[1] = pack8(f1);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = tid + 256 * i, jv = e >> 4, d4 = 4 * (e & 15);
        vs[jv][d4] = vx[i].x;
        vs[jv][d4 + 1] = vx[i].y;
        vs[jv][d4 + 2] = vx[i].z;
        vs[jv][d4 + 3] = vx[i].w;
    }
    __syncthreads();
    for (int e = tid; e < kD * 8; e += 256) {
        const int d = e >> 3, c = e & 7;
        float v[8], lo[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = vs[8 * c + q][d];
        const uint4 hi = pack8(v);
        const uint32_t hw[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hw[q]));
            lo[2 * q] = v[2 * q] - b.x;
            lo[2 * q + 1] = v[2 * q + 1] - b.y;
        }
        __half* row_h = a.att_vt + ((head * 2 + 0) * kD + d) * a.n_ctx64 + j0 + 8 * c;
        __half* row_l = a.att_vt + ((head * 2 + 1) * kD + d) * a.n_ctx64 + j0 + 8 * c;
        const uint4 lw = pack8(lo);
        if (j0 + 8 * c + 8 <= end) {
            *reinterpret_cast<uint4*>(row_h) = hi;
            *reinterpret_cast<uint4*>(row_l) = lw;
        } else {
            // The last keys below seq_conv: the ones past it are the QKV
            // epilogue's (this call's rows) and stay as written.
            const __half* hh = reinterpret_cast<const __half*>(&hi);
            const __half* ll = reinterpret_cast<const __half*>(&lw);
            for (int q = 0; j0 + 8 * c + q < end; ++q) {
                row_h[q] = hh[q];
                row_l[q] = ll[q];
            }
        }
    }
}

// ---- attention -------------------------------------------------------------------

// Shared memory (1024-byte aligned; every operand tile has 128-byte rows in
// the 128-byte swizzle).
struct TcAttnSmem {
    unsigned char q[kRows * 128];
    unsigned char p[kRows * 128];
    unsigned char kv[kStages][3][kTileBytes];  // per stage: K, V^T hi, V^T lo
    float part[2][kRows];                      // per row: the two threads' partial max (then sum)
    uint64_t full[kStages], bar_s, bar_o;
    uint32_t tmem_slot;
    int abort;
};
constexpr size_t kSmemBytes = sizeof(TcAttnSmem) + 1024;

// Byte offset of the 16-byte chunk c (elements 8c .. 8c + 7) of row r in a
// tile of 128-byte rows with the 128-byte swizzle: chunk c ^ (r mod 8).
__device__ __forceinline__ uint32_t sw_chunk(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive f32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 2^x by the MUFU instruction (relative error about 2^-22, flushes
// subnormal results to zero: the probabilities then enter the MMAs as f16).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// One lane of the warp waits on `bar`; the warp follows its verdict.  A wait
// that runs out marks the block aborted and raises the guard word.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, unsigned par, int* abort_flag, int* err) {
    int got = 1;
    if ((threadIdx.x & 31) == 0) got = sm100::mbar_wait(bar, par, kWaitNs) ? 1 : 0;
    got = __shfl_sync(0xffffffffu, got, 0);
    if (!got && (threadIdx.x & 31) == 0) {
        *abort_flag = 1;
        raise_guard(err, kGuardTimeout);
    }
    return got != 0;
}

__device__ __forceinline__ void block_sync_tc() {
    sm100::tc_fence_before();
    __syncthreads();
    sm100::tc_fence_after();
}

// The two warps w and w + 4 (the two threads of every row they own).
__device__ __forceinline__ void pair_sync(int warp) {
    asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
}

__global__ void __launch_bounds__(kThreads, 2)
    k_attn_prefill_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_vt,
                      PrefillAttnArgs a, int layer, int n_ctx64, int* err) {
    using namespace sm100;
    extern __shared__ unsigned char pt_smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(pt_smem_raw) & 1023u)) & 1023u;
    TcAttnSmem& sm = *reinterpret_cast<TcAttnSmem*>(pt_smem_raw + pad);
    const int g = blockIdx.x, blk = blockIdx.y;
    const int r0 = a.blk_row0[blk], nr = a.blk_nrows[blk];
    const int group = a.nh / a.nkv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot = a.slot[r0];
    // Largest position of the block's rows.
    int pmax = lane < nr ? a.pos[r0 + lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
    const int n_tiles = pmax / kKT + 1;
    const int head = slot * a.nkv + g;
    const int k_row0 = head * n_ctx64, vt_row0 = head * 2 * kD;
    const bool issuer = warp == 4 && lane == 0;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[s], 1);
        mbar_init(&sm.bar_s, 1);
        mbar_init(&sm.bar_o, 1);
        mbar_init_fence();
        sm.abort = 0;
    }
    if (issuer) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_vt);
    }
    if (warp == 4) tmem_alloc(&sm.tmem_slot, kTmemCols);
    // Launched with programmatic stream serialisation: the set-up above
    // overlaps the previous kernel; q and the operands are read only after it.
    pdl_launch_dependents();
    pdl_wait();
    // Q: 128 rows x 8 chunks, four chunks per thread, f32 -> f16.
    for (int e = tid; e < kRows * 8; e += kThreads) {
        const int r = e >> 3, c = e & 7, i = r / group, h = r % group;
        float f[8];
        if (i < nr) {
            const float* src = a.q + (size_t)(r0 + i) * a.nh * kD + (size_t)(g * group + h) * kD + 8 * c;
            const float4 x0 = *reinterpret_cast<const float4*>(src);
            const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
            f[0] = x0.x; f[1] = x0.y; f[2] = x0.z; f[3] = x0.w;
            f[4] = x1.x; f[5] = x1.y; f[6] = x1.z; f[7] = x1.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = 0.f;
        }
        *reinterpret_cast<uint4*>(sm.q + sw_chunk(r, c)) = pack8(f);
    }
    fence_async_smem();
    block_sync_tc();
    const uint32_t tmem = sm.tmem_slot;
    // S in columns 0-63; the value products of even and odd tiles in 64-127
    // and 128-191.
    const uint32_t t_s = tmem, t_o = tmem + kKT;
    constexpr uint32_t idesc = idesc_f16_f32(kRows, kKT);

    // Issuer-side state: tiles whose copies were issued / seen complete.
    int n_loaded = 0, n_landed = 0;
    auto load_tile = [&](int t) {
        const int s = t % kStages;
        mbar_expect_tx(&sm.full[s], 3 * kTileBytes);
        tma_load_2d(sm.kv[s][0], &tm_k, 0, k_row0 + t * kKT, &sm.full[s]);
        tma_load_2d(sm.kv[s][1], &tm_vt, t * kKT, vt_row0, &sm.full[s]);
        tma_load_2d(sm.kv[s][2], &tm_vt, t * kKT, vt_row0 + kD, &sm.full[s]);
        ++n_loaded;
    };
    // S(t) = Q . K_t^T once tile t has landed.
    auto issue_s = [&](int t) {
        const int s = t % kStages;
        if (!mbar_wait(&sm.full[s], (unsigned)((t / kStages) & 1), kWaitNs)) {
            sm.abort = 1;
            raise_guard(err, kGuardTimeout);
            return;
        }
        ++n_landed;
        tc_fence_after();
        const uint64_t qd = desc_sw128(smem_addr(sm.q)), kd = desc_sw128(smem_addr(sm.kv[s][0]));
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) mma_f16(t_s, qd + 2 * k, kd + 2 * k, idesc, k != 0 ? 1u : 0u);
        mma_commit(&sm.bar_s);
    };
    if (issuer) {
        load_tile(0);
        if (n_tiles > 1) load_tile(1);
        issue_s(0);
    }

    // The row this thread owns and its half of the columns.
    const int row = 32 * (warp & 3) + lane, half = warp >> 2;
    const int ri = row / group, rh = row % group;
    const bool rvalid = ri < nr;
    const int prow = rvalid ? a.pos[r0 + ri] : -1;
    const uint32_t tl = (uint32_t)(32 * (warp & 3)) << 16;  // this warp's TMEM lane offset
    const uint32_t ts = t_s + tl + 32 * half, to = t_o + tl + 32 * half;  // + 64 for odd tiles
    float o_acc[kD / 2];
#pragma unroll
    for (int d = 0; d < kD / 2; ++d) o_acc[d] = 0.f;
    float m_run = -INFINITY, l_run = 0.f, corr_prev = 1.f;

    // o_acc = o_acc * corr + O_t (the value product of tile t_prev, which
    // this thread has seen complete).
    auto fold = [&](int t_prev, float corr) {
        const uint32_t src = to + (uint32_t)(kKT * (t_prev & 1));
#pragma unroll
        for (int h16 = 0; h16 < 2; ++h16) {
            float v[16];
            tmem_ld16(src + 16 * h16, v);
#pragma unroll
            for (int c = 0; c < 16; ++c) o_acc[16 * h16 + c] = fmaf(o_acc[16 * h16 + c], corr, v[c]);
        }
    };

    int t = 0;
    for (; t < n_tiles; ++t) {
        const int jh = t * kKT + 32 * half;  // first key of this thread's columns
        // ---- row maximum of S(t) over the keys this row sees ---------------
        // Columns past the row's position are masked; a tile wholly at or
        // below the diagonal (for this thread's columns) needs no mask.
        const bool got_s = warp_wait(&sm.bar_s, (unsigned)(t & 1), &sm.abort, err);
        const bool full_cols = jh + 31 <= prow;
        float v[32];
        float mx = -INFINITY;
        if (got_s) {
            tc_fence_after();
            tmem_ld32(ts, v);
            if (!full_cols) {
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (jh + c > prow) v[c] = -INFINITY;
            }
            float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
            for (int c = 4; c < 32; ++c) m4[c & 3] = fmaxf(m4[c & 3], v[c]);
            mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        }
        // Every thread of both warps passes this barrier, whatever its wait returned.
        sm.part[half][row] = mx;
        pair_sync(warp);
        mx = fmaxf(mx, sm.part[half ^ 1][row]);
        const float m_new = rvalid ? fmaxf(m_run, mx) : 0.f;
        const float corr = (rvalid && m_run != -INFINITY) ? ex2((m_run - m_new) * kScaleLog2) : 0.f;
        // ---- probabilities of this tile to shared memory -----------------------
        // P is free once the previous tile's value product has completed.
        const bool p_free = t == 0 || warp_wait(&sm.bar_o, (unsigned)((t - 1) & 1), &sm.abort, err);
        if (got_s && p_free) {
            const float mb = -m_new * kScaleLog2;
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                v[c] = rvalid ? ex2(fmaf(v[c], kScaleLog2, mb)) : 0.f;  // ex2(-inf) = 0
                l4[c & 3] += v[c];
            }
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
                const float f[8] = {v[8 * c8], v[8 * c8 + 1], v[8 * c8 + 2], v[8 * c8 + 3],
                                    v[8 * c8 + 4], v[8 * c8 + 5], v[8 * c8 + 6], v[8 * c8 + 7]};
                *reinterpret_cast<uint4*>(sm.p + sw_chunk(row, 4 * half + c8)) = pack8(f);
            }
            if (rvalid) {
                l_run = l_run * corr + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
                m_run = m_new;
            }
        }
        fence_async_smem();
        block_sync_tc();
        if (sm.abort) break;
        // ---- next scores, this tile's value product, the copy two tiles on ----
        // S is free (every thread has read it), and so is the stage of tile
        // t - 1 (every thread has waited for its value product).
        if (issuer) {
            if (t + 1 < n_tiles) issue_s(t + 1);
            const int s = t % kStages;
            const uint32_t d = t_o + (uint32_t)(kKT * (t & 1));
            const uint64_t pd = desc_sw128(smem_addr(sm.p));
            const uint64_t hd = desc_sw128(smem_addr(sm.kv[s][1])), ld = desc_sw128(smem_addr(sm.kv[s][2]));
#pragma unroll
            for (int k = 0; k < kKT / 16; ++k) mma_f16(d, pd + 2 * k, hd + 2 * k, idesc, k != 0 ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < kKT / 16; ++k) mma_f16(d, pd + 2 * k, ld + 2 * k, idesc, 1u);
            mma_commit(&sm.bar_o);
            if (t + 2 < n_tiles) load_tile(t + 2);
        }
        // ---- the previous tile's value product, while the MMAs run ---------
        // (every thread waited for it before writing P; a second wait on its
        // phase here could alias the phase of the product just issued)
        if (t > 0) fold(t - 1, corr_prev);
        corr_prev = corr;
    }
    if (t == n_tiles && warp_wait(&sm.bar_o, (unsigned)((n_tiles - 1) & 1), &sm.abort, err)) {
        tc_fence_after();
        fold(n_tiles - 1, corr_prev);
    }
    sm.part[half][row] = l_run;
    block_sync_tc();
    // ---- output: o / l as the f16 hi / lo pair ---------------------------------
    if (rvalid && !sm.abort) {
        const float inv = 1.f / (l_run + sm.part[half ^ 1][row]);
        const size_t off = (size_t)(r0 + ri) * a.nh * kD + (size_t)(g * group + rh) * kD + 32 * half;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float hi[8], lo[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float x = o_acc[8 * c + q] * inv;
                hi[q] = __half2float(__float2half_rn(x));
                lo[q] = x - hi[q];
            }
            *reinterpret_cast<uint4*>(a.o_h + off + 8 * c) = pack8(hi);
            *reinterpret_cast<uint4*>(a.o_l + off + 8 * c) = pack8(lo);
        }
    }
    // A block that stopped early may still have tiles in flight: let them
    // land before the shared memory is released.
    if (issuer)
        for (int j = n_landed; j < n_loaded; ++j)
            if (!mbar_wait(&sm.full[j % kStages], (unsigned)((j / kStages) & 1), kWaitNs)) {
                raise_guard(err, kGuardTimeout);
                break;
            }
    if (warp == 4) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t enqueue_attn_prefill_tc(const Ctx& c, const PrefillAttnArgs& a, const PrefillPlan& plan, int layer,
                                    cudaStream_t st) {
    const int n64 = att_ctx64(a.n_ctx);
    if (plan.conv_tiles > 0) {
        OperandArgs oa{a.kv, plan.seq_slot, plan.seq_conv, c.ws.att_k, c.ws.att_vt, a.nkv, a.n_ctx, n64, a.L,
                       layer};
        cudaError_t e = launch_pdl(k_att_operands, dim3(plan.conv_tiles, plan.n_seq, a.nkv), dim3(256), 0, st, oa);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(k_attn_prefill_tc, dim3(a.nkv, plan.n_blk), dim3(kThreads), kSmemBytes, st, c.tc.att_k,
                      c.tc.att_vt, a, layer, n64, c.err);
}

cudaError_t prefill_attn_tc_set_smem() {
    return cudaFuncSetAttribute(k_attn_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
}

}  // namespace qwen2
