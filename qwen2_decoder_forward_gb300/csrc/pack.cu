// Weight-layout packer, Q8_0 quantiser and RoPE table (host side).
#include <math.h>
#include <string.h>

#include <vector>

#include "ctx.h"

namespace qwen2 {

namespace {

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

float h2f(uint16_t b) {
    __half_raw r;
    r.x = b;
    return __half2float(__half(r));
}
uint16_t f2h(float f) {
    __half_raw r = static_cast<__half_raw>(__float2half_rn(f));
    return r.x;
}

struct Blob {
    char* host_base;
    char* dev_base;
    size_t off = 0;
    char* take(size_t bytes, char** dev) {
        off = align_up(off, 256);
        char* h = host_base + off;
        *dev = dev_base + off;
        off += bytes;
        return h;
    }
};

// Place one matrix whose host rows come from `row_src(r)` (an f16 row of k
// values) into the blob, in f16 or Q8_0.
template <class RowSrc>
DevMat put_mat(Blob& b, int rows, int k, int fmt, RowSrc row_src) {
    DevMat m;
    m.rows = rows;
    m.k = k;
    if (fmt == QWEN2_WEIGHTS_Q4_0) {
        char* dq;
        uint8_t* hq = reinterpret_cast<uint8_t*>(b.take((size_t)rows * (k / 2), &dq));
        char* dd;
        uint16_t* hd = reinterpret_cast<uint16_t*>(b.take((size_t)rows * (k / 32) * 2, &dd));
        for (int r = 0; r < rows; ++r)
            quantize_q4_0_host(row_src(r), 1, k, hq + (size_t)r * (k / 2), hd + (size_t)r * (k / 32));
        m.q = reinterpret_cast<const int8_t*>(dq);
        m.d = reinterpret_cast<const __half*>(dd);
        m.q4 = true;
    } else if (fmt == QWEN2_WEIGHTS_Q8_0) {
        char* dq;
        int8_t* hq = reinterpret_cast<int8_t*>(b.take((size_t)rows * k, &dq));
        char* dd;
        uint16_t* hd = reinterpret_cast<uint16_t*>(b.take((size_t)rows * (k / 32) * 2, &dd));
        for (int r = 0; r < rows; ++r)
            quantize_q8_0_host(row_src(r), 1, k, hq + (size_t)r * k, hd + (size_t)r * (k / 32));
        m.q = reinterpret_cast<const int8_t*>(dq);
        m.d = reinterpret_cast<const __half*>(dd);
    } else {
        char* dw;
        uint16_t* hw = reinterpret_cast<uint16_t*>(b.take((size_t)rows * k * 2, &dw));
        for (int r = 0; r < rows; ++r) memcpy(hw + (size_t)r * k, row_src(r), (size_t)k * 2);
        m.w = reinterpret_cast<const __half*>(dw);
    }
    return m;
}

const float* put_f32(Blob& b, const float* src, size_t n) {
    char* d;
    float* h = reinterpret_cast<float*>(b.take(n * 4, &d));
    memcpy(h, src, n * 4);
    return reinterpret_cast<const float*>(d);
}

// Original row of packed Q/K/V row `pr`: within each head slot of hd rows,
// packed rows (2i, 2i+1) hold original rows (i, i + hd/2).
int qkv_orig_row(int pr, int hd) {
    const int s = pr / hd, within = pr % hd;
    return s * hd + (within >> 1) + (within & 1) * (hd / 2);
}

}  // namespace

void quantize_q8_0_host(const uint16_t* w, int64_t rows, int64_t k, int8_t* q, uint16_t* d) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < k / 32; ++b) {
            const uint16_t* x = w + r * k + b * 32;
            float amax = 0.f;
            for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(h2f(x[e])));
            const float dd = amax / 127.0f;
            int8_t* qq = q + r * k + b * 32;
            for (int e = 0; e < 32; ++e) {
                if (dd == 0.f) {
                    qq[e] = 0;
                    continue;
                }
                float v = roundf(h2f(x[e]) / dd);  // half away from zero
                v = fminf(127.f, fmaxf(-127.f, v));
                qq[e] = (int8_t)v;
            }
            d[r * (k / 32) + b] = f2h(dd);
        }
    }
}

// Q4_0 (the four-bit counterpart of the Q8_0 reading): blocks of 32 along
// k; d = max|x| / 7 in f32; c = clamp(round-half-away(x / d), -7, 7) (c = 0
// where d = 0), stored as the nibble c + 8, element 2j in the low nibble of
// byte j; the stored scale is f16(d), round to nearest even.
void quantize_q4_0_host(const uint16_t* w, int64_t rows, int64_t k, uint8_t* packed, uint16_t* d) {
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < k / 32; ++b) {
            const uint16_t* x = w + r * k + b * 32;
            float amax = 0.f;
            for (int e = 0; e < 32; ++e) amax = fmaxf(amax, fabsf(h2f(x[e])));
            const float dd = amax / 7.0f;
            uint8_t* pp = packed + r * (k / 2) + b * 16;
            for (int e = 0; e < 32; e += 2) {
                int c[2] = {0, 0};
                for (int i = 0; i < 2; ++i) {
                    if (dd == 0.f) continue;
                    float v = roundf(h2f(x[e + i]) / dd);  // half away from zero
                    v = fminf(7.f, fmaxf(-7.f, v));
                    c[i] = (int)v;
                }
                pp[e / 2] = (uint8_t)((c[0] + 8) | ((c[1] + 8) << 4));
            }
            d[r * (k / 32) + b] = f2h(dd);
        }
    }
}

int pack_weights(Ctx& c, const qwen2_weights* w, std::string& err) {
    const qwen2_config& g = c.cfg;
    const int H = g.hidden, I = g.intermediate, V = g.vocab, hd = g.head_dim;
    const int nq = g.n_head * hd, nkv = g.n_kv_head * hd;
    const int fmt = g.weight_format;
    c.nqkv = nq + 2 * nkv;

    size_t total = 0;
    auto add = [&](size_t bytes) { total = align_up(total, 256) + bytes; };
    auto add_mat = [&](int rows, int k) {
        if (fmt == QWEN2_WEIGHTS_Q4_0) {
            add((size_t)rows * (k / 2));
            add((size_t)rows * (k / 32) * 2);
        } else if (fmt == QWEN2_WEIGHTS_Q8_0) {
            add((size_t)rows * k);
            add((size_t)rows * (k / 32) * 2);
        } else {
            add((size_t)rows * k * 2);
        }
    };
    add_mat(V, H);
    if (w->lm_head) add_mat(V, H);
    add((size_t)H * 4);
    for (int l = 0; l < g.n_layer; ++l) {
        add_mat(c.nqkv, H);
        add_mat(H, nq);
        add_mat(2 * I, H);
        add_mat(H, I);
        add((size_t)c.nqkv * 4);
        add((size_t)H * 4);
        add((size_t)H * 4);
    }
    total = align_up(total, 256);

    std::vector<char> host(total, 0);
    if (cudaMalloc(&c.wblob, total) != cudaSuccess) {
        cudaGetLastError();
        c.wblob = nullptr;
        err = "cudaMalloc of " + std::to_string(total) + " weight bytes failed";
        return QWEN2_E_OOM;
    }
    c.wbytes = total;
    Blob b{host.data(), static_cast<char*>(c.wblob)};

    c.embed = put_mat(b, V, H, fmt, [&](int r) { return w->embed + (size_t)r * H; });
    c.lm_head = w->lm_head ? put_mat(b, V, H, fmt, [&](int r) { return w->lm_head + (size_t)r * H; }) : c.embed;
    c.final_norm = put_f32(b, w->final_norm, H);
    c.layers.resize(g.n_layer);
    std::vector<float> bperm(c.nqkv);
    for (int l = 0; l < g.n_layer; ++l) {
        const qwen2_layer_weights& L = w->layers[l];
        DevLayer& D = c.layers[l];
        auto qkv_src = [&](int pr) -> const uint16_t* {
            const int orig = qkv_orig_row(pr, hd);
            if (orig < nq) return L.wq + (size_t)orig * H;
            if (orig < nq + nkv) return L.wk + (size_t)(orig - nq) * H;
            return L.wv + (size_t)(orig - nq - nkv) * H;
        };
        D.wqkv = put_mat(b, c.nqkv, H, fmt, qkv_src);
        for (int pr = 0; pr < c.nqkv; ++pr) {
            const int orig = qkv_orig_row(pr, hd);
            bperm[pr] = orig < nq ? L.bq[orig] : orig < nq + nkv ? L.bk[orig - nq] : L.bv[orig - nq - nkv];
        }
        D.wo = put_mat(b, H, nq, fmt, [&](int r) { return L.wo + (size_t)r * nq; });
        D.wgu = put_mat(b, 2 * I, H, fmt, [&](int r) {
            return (r & 1) ? L.wu + (size_t)(r >> 1) * H : L.wg + (size_t)(r >> 1) * H;
        });
        D.wd = put_mat(b, H, I, fmt, [&](int r) { return L.wd + (size_t)r * I; });
        D.bqkv = put_f32(b, bperm.data(), c.nqkv);
        D.attn_norm = put_f32(b, L.attn_norm, H);
        D.ffn_norm = put_f32(b, L.ffn_norm, H);
    }
    if (b.off > total) {
        err = "packer size mismatch";
        return QWEN2_E_CUDA;
    }
    if (cudaMemcpy(c.wblob, host.data(), total, cudaMemcpyHostToDevice) != cudaSuccess) {
        err = "weight upload failed";
        return QWEN2_E_CUDA;
    }
    return QWEN2_OK;
}

int build_rope_table(Ctx& c, std::string& err) {
    const int n = c.cfg.n_ctx, half = c.cfg.head_dim / 2;
    std::vector<float2> t((size_t)n * half);
    for (int i = 0; i < half; ++i) {
        const double inv = pow(c.cfg.rope_theta, -2.0 * i / c.cfg.head_dim);
        for (int p = 0; p < n; ++p) {
            const double a = (double)p * inv;
            t[(size_t)p * half + i] = make_float2((float)cos(a), (float)sin(a));
        }
    }
    if (cudaMalloc(&c.rope, t.size() * sizeof(float2)) != cudaSuccess) {
        cudaGetLastError();
        c.rope = nullptr;
        err = "cudaMalloc of the RoPE table failed";
        return QWEN2_E_OOM;
    }
    if (cudaMemcpy(c.rope, t.data(), t.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
        err = "RoPE table upload failed";
        return QWEN2_E_CUDA;
    }
    return QWEN2_OK;
}

}  // namespace qwen2
