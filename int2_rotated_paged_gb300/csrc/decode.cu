// decode.cu -- read path of the INT2 rotated paged KV cache (sm_103a): paged GQA decode
// attention over INT2 pages + BF16 sink / window tokens, split over the context with a
// log-sum-exp combine.
//
// The pages' read path (axbrief.com OSCAR page, section "attention-statistics rotation +
// Triton kernels") unpacks, dequantises and inverse-rotates the keys inside one fused
// attention pass.  Here the rotation is applied once to the query (q~ = q . R_K), which
// equals inverse-rotating every key because R_K is orthogonal; keys and values are
// dequantised in registers (x^ = m + code * s, folded into the dot products) and never
// written back.
//
// Kernels:
//   rotate_q      q~ = q . R_K for every (request, query head), fp32.
//   split_simt    one CTA per (split, KV head, request): online softmax over its INT2
//                 pages (or, for the last split of a request, over the BF16 tokens) for
//                 the G query heads of the KV head; writes (max, sum, unnormalised out).
//   combine       out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s per (request, head).
//   combine_mma   the same merge for the warp-MMA path (prep.cu, decode_mma.cu): the BF16
//                 partial and the partials of the warps that streamed the request's pages.
// launch_decode runs either path; launch_decode_step runs the fused decode step
// (prep_step -> decode_mma -> combine_mma).
// All softmax arithmetic is in base 2 (logits pre-scaled by log2(e) / sqrt(128)).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace oscar {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }
__device__ __forceinline__ float h2f(uint16_t b) { return __half2float(__ushort_as_half(b)); }

__device__ __forceinline__ float load_q(const DecodeParams& p, size_t idx) {
    return p.q_dtype == 0 ? reinterpret_cast<const float*>(p.q)[idx]
                          : bf16f(reinterpret_cast<const uint16_t*>(p.q)[idx]);
}

// q~[b][hq][c] = sum_j q[b][hq][j] R_{hq / G}[j][c]
__global__ void __launch_bounds__(128) rotate_q(const __grid_constant__ DecodeParams p) {
    __shared__ float qs[kMaxG][kD];
    const int b = blockIdx.y;
    const int h = blockIdx.x;
    const int c = threadIdx.x;
    if (b == 0 && h == 0 && c == 0 && p.err) *p.err = 0;
    const size_t qbase = ((size_t)b * p.hkv * p.g + (size_t)h * p.g) * kD;
    for (int i = 0; i < p.g; ++i) qs[i][c] = load_q(p, qbase + (size_t)i * kD + c);
    __syncthreads();
    float acc[kMaxG];
#pragma unroll
    for (int i = 0; i < kMaxG; ++i) acc[i] = 0.f;
    // column c of R_h, 32 rows at a time so that the loads are in flight together
    const float* R = p.rk + (size_t)h * kD * kD + c;
    for (int j0 = 0; j0 < kD; j0 += 32) {
        float r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __ldg(R + (size_t)(j0 + j) * kD);
#pragma unroll
        for (int j = 0; j < 32; ++j)
#pragma unroll
            for (int i = 0; i < kMaxG; ++i)
                if (i < p.g) acc[i] = fmaf(qs[i][j0 + j], r[j], acc[i]);
    }
    for (int i = 0; i < p.g; ++i) p.qrot[qbase + (size_t)i * kD + c] = acc[i];
}

template <int G>
struct WarpState {
    float m[G], l[G], o[G][4];
};

template <int G>
__device__ __forceinline__ void softmax_update(WarpState<G>& st, const float (&lg)[4][G],
                                               const float (&vv)[4][4]) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        float mx = st.m[hh];
#pragma unroll
        for (int i = 0; i < 4; ++i) mx = fmaxf(mx, lg[i][hh]);
        const float sc = exp2f(st.m[hh] - mx);   // 0 when m was -inf
        float pi[4];
        float ps = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            pi[i] = exp2f(lg[i][hh] - mx);
            ps += pi[i];
        }
        st.l[hh] = st.l[hh] * sc + ps;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float a = st.o[hh][j] * sc;
#pragma unroll
            for (int i = 0; i < 4; ++i) a = fmaf(pi[i], vv[i][j], a);
            st.o[hh][j] = a;
        }
        st.m[hh] = mx;
    }
}

template <int G>
__global__ void __launch_bounds__(128) split_simt(const __grid_constant__ DecodeParams p) {
    __shared__ float sm_m[4][G], sm_l[4][G];
    __shared__ float sm_o[4][G][kD];
    const int b = blockIdx.z;
    const int h = blockIdx.y;
    const int len = p.len[b];
    if (len == 0) return;
    const int nsp = int2_splits(len, p.pps);
    const int s = (int)blockIdx.x;
    if (s > nsp) return;
    const int w = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool bf16_split = (s == nsp);
    const float qscale = kLog2e * rsqrtf((float)kD);

    // This lane's 4 query channels (rotated for INT2 tokens, plain for BF16) and 4 output
    // channels.  INT2: the key channels whose codes share byte `lane` of a token row (bits 2j)
    // and the value channels whose codes share one byte of the value region; BF16: 4 lane + j.
    auto kch = [&](int j) {
        return bf16_split ? 4 * lane + j
                          : 64 * ((lane >> 2) & 1) + 16 * j + 8 * (lane & 1) + 2 * (lane >> 3) + ((lane >> 1) & 1);
    };
    auto och = [&](int j) { return bf16_split ? 4 * lane + j : 64 * (lane >> 4) + 16 * j + 8 * ((lane >> 3) & 1) + (lane & 7); };
    float qr[G][4];
    float qsum[G];   // sum of this lane's 4 rotated channels (for the m * sum(q) term)
    const size_t qbase = ((size_t)b * p.hkv * p.g + (size_t)h * p.g) * kD;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        qsum[hh] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const size_t idx = qbase + (size_t)hh * kD + kch(j);
            qr[hh][j] = (bf16_split ? load_q(p, idx) : p.qrot[idx]) * qscale;
            qsum[hh] += qr[hh][j];
        }
    }
    WarpState<G> st;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        st.m[hh] = -INFINITY;
        st.l[hh] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) st.o[hh][j] = 0.f;
    }

    if (!bf16_split) {
        const int n_tok = int2_tokens(len);
        const int pg_end = min((s + 1) * p.pps, int2_pages(len));
        const int kgrp = (lane >> 2) & 1;   // group of this lane's key channels
        const int vgrp = lane >> 4;         // group of this lane's value channels
        for (int pg = s * p.pps + w; pg < pg_end; pg += 4) {
            const int phys = p.page_table[(size_t)b * p.max_pps + pg];
            const uint8_t* blk = p.pool + ((size_t)phys * p.hkv + h) * p.fmt.bytes;
            const int nt = min(kPage, n_tok - pg * kPage);
            for (int t4 = 0; t4 < nt; t4 += 4) {
                float lg[4][G];
                float vv[4][4];
                // V: one byte per token holds this lane's 4 value channels (bits 2j)
                uint32_t vb[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) vb[i] = blk[p.fmt.v_codes + v_code_byte(t4 + i, och(0))];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int t = t4 + i;
                    const uint32_t kb = blk[kKCodes + t * 32 + lane];
                    const uint32_t ksm =
                        *reinterpret_cast<const uint32_t*>(blk + p.fmt.k_sm + t * p.fmt.k_stride + (p.fmt.gk == 64 ? kgrp * 4 : 0));
                    const uint32_t vsm =
                        *reinterpret_cast<const uint32_t*>(blk + p.fmt.v_sm + t * p.fmt.v_stride + (p.fmt.gv == 64 ? vgrp * 4 : 0));
                    const float ks = h2f(ksm & 0xffff), km = h2f(ksm >> 16);
                    const float vs = h2f(vsm & 0xffff), vm = h2f(vsm >> 16);
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        float d = 0.f;
#pragma unroll
                        for (int j = 0; j < 4; ++j) d = fmaf(qr[hh][j], (float)((kb >> (2 * j)) & 3), d);
                        lg[i][hh] = fmaf(ks, d, km * qsum[hh]);
                    }
                    // slots past the request's last token hold stale bytes (possibly NaN
                    // scales): their values must be exact zeros, not 0 * garbage
                    const bool live = t < nt;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        vv[i][j] = live ? fmaf((float)((vb[i] >> (2 * j)) & 3), vs, vm) : 0.f;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        float x = lg[i][hh];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                        lg[i][hh] = (t4 + i < nt) ? x : -INFINITY;
                    }
                softmax_update<G>(st, lg, vv);
            }
        }
    } else {
        // BF16 tokens: sink slots [0, n_sink) and window slots [sink, sink + n_win)
        const int n_sink = min(len, kSink);
        const int n_win = min(kWindow, max(0, len - kSink));
        const int n_all = n_sink + n_win;
        const uint16_t* kb = p.bf16 + (((size_t)b * p.hkv + h) * 2 + 0) * kSlots * kD;
        const uint16_t* vb = p.bf16 + (((size_t)b * p.hkv + h) * 2 + 1) * kSlots * kD;
        for (int t4 = 4 * w; t4 < n_all; t4 += 16) {
            float lg[4][G];
            float vv[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = min(t4 + i, n_all - 1);
                const int slot = t < n_sink ? t : kSink + (t - n_sink);
                const uint2 kr = *reinterpret_cast<const uint2*>(kb + (size_t)slot * kD + 4 * lane);
                const uint2 vr = *reinterpret_cast<const uint2*>(vb + (size_t)slot * kD + 4 * lane);
                const float kf[4] = {bf16f(kr.x & 0xffff), bf16f(kr.x >> 16), bf16f(kr.y & 0xffff),
                                     bf16f(kr.y >> 16)};
                vv[i][0] = bf16f(vr.x & 0xffff);
                vv[i][1] = bf16f(vr.x >> 16);
                vv[i][2] = bf16f(vr.y & 0xffff);
                vv[i][3] = bf16f(vr.y >> 16);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float d = 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) d = fmaf(qr[hh][j], kf[j], d);
                    lg[i][hh] = d;
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float x = lg[i][hh];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
                    lg[i][hh] = (t4 + i < n_all) ? x : -INFINITY;
                }
            softmax_update<G>(st, lg, vv);
        }
    }

    // merge the 4 warps and write this split's partial result
    if (lane == 0) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            sm_m[w][hh] = st.m[hh];
            sm_l[w][hh] = st.l[hh];
        }
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
#pragma unroll
        for (int j = 0; j < 4; ++j) sm_o[w][hh][och(j)] = st.o[hh][j];
    __syncthreads();
    const int c = threadIdx.x;
    float* part = p.partial + (((size_t)b * p.hkv + h) * p.max_splits + s) * p.g * (2 + kD);
    for (int hh = 0; hh < G; ++hh) {
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < 4; ++ww) M = fmaxf(M, sm_m[ww][hh]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int ww = 0; ww < 4; ++ww) {
            const float f = sm_m[ww][hh] == -INFINITY ? 0.f : exp2f(sm_m[ww][hh] - M);
            L = fmaf(f, sm_l[ww][hh], L);
            O = fmaf(f, sm_o[ww][hh][c], O);
        }
        float* ph = part + (size_t)hh * (2 + kD);
        if (c == 0) {
            ph[0] = M;
            ph[1] = L;
        }
        ph[2 + c] = O;
    }
}

__device__ __forceinline__ void merge(const float* ph, int c, float& M, float& L, float& O) {
    const float m = ph[0];
    if (m == -INFINITY) return;
    const float nm = fmaxf(M, m);
    const float fa = M == -INFINITY ? 0.f : exp2f(M - nm);
    const float fb = exp2f(m - nm);
    L = L * fa + ph[1] * fb;
    O = O * fa + ph[2 + c] * fb;
    M = nm;
}

__global__ void __launch_bounds__(128) combine(const __grid_constant__ DecodeParams p) {
    const int b = blockIdx.y;
    const int hq = blockIdx.x;
    const int h = hq / p.g;
    const int hh = hq % p.g;
    const int c = threadIdx.x;
    const int len = p.len[b];
    const size_t oidx = ((size_t)b * p.hkv * p.g + hq) * kD + c;
    float res = 0.f;
    if (len > 0) {
        float M = -INFINITY, L = 0.f, O = 0.f;
        {
            const int ns = int2_splits(len, p.pps) + 1;
            const float* part = p.partial + ((size_t)b * p.hkv + h) * p.max_splits * p.g * (2 + kD);
            for (int s = 0; s < ns; ++s) merge(part + ((size_t)s * p.g + hh) * (2 + kD), c, M, L, O);
        }
        res = O / L;
    }
    if (p.out_dtype == 0)
        reinterpret_cast<float*>(p.out)[oidx] = res;
    else
        reinterpret_cast<__nv_bfloat16*>(p.out)[oidx] = __float2bfloat16_rn(res);
}

// Warp-MMA path: one CTA per (KV head, request), one warp per query head, lane = channels
// 2 lane, 2 lane + 1, 64 + 2 lane, 65 + 2 lane.  Merges the BF16 partial with the partials of the
// warps w0 .. w1 that owned pages of (b, h) (warps whose page range is empty wrote nothing).  Lane i
// reads the reference max and sum of partial w0 + i (and further ones 32 apart), so the common max
// and the total sum are warp reductions; the unnormalised outputs are then summed four partials at a
// time, every load independent of the merge.
__global__ void __launch_bounds__(32 * kMaxG) combine_mma(const __grid_constant__ DecodeParams p) {
    const int h = blockIdx.x, b = blockIdx.y;
    const int hh = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int len = p.len[b];
    const int u = b * p.hkv + h;
    float2 r0 = make_float2(0.f, 0.f), r1 = r0;
    if (len > 0) {
        const float* pb = p.part_bf16 + ((size_t)u * p.g + hh) * (2 + kD);
        const int pages = int2_pages(len);
        int w0 = 0, w1 = -1;
        if (pages > 0) {
            const int pf = p.page_off[b] + h * pages;
            w0 = (int)((((long long)pf + 1) * p.n_units - 1) / p.total_pages);
            w1 = (int)((((long long)pf + pages) * p.n_units - 1) / p.total_pages);
        }
        auto slot = [&](int w) { return p.part_mma + (((size_t)u + w) * p.g + hh) * (2 + kD); };
        auto owns = [&](int w) {
            return ((long long)w * p.total_pages) / p.n_units != ((long long)(w + 1) * p.total_pages) / p.n_units;
        };
        const int n = w1 - w0 + 1;   // candidate partials (those of warps that own no page are skipped)
        // common max: the BF16 partial's and every owned INT2 partial's reference max
        float M = pb[0];
        for (int i = lane; i < n; i += 32)
            if (owns(w0 + i)) M = fmaxf(M, slot(w0 + i)[0]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.f;
        float2 o0 = r0, o1 = r0;
        auto add = [&](const float* ph, float f) {
            const float2 a = *reinterpret_cast<const float2*>(ph + 2 + 2 * lane);
            const float2 c = *reinterpret_cast<const float2*>(ph + 2 + 64 + 2 * lane);
            o0 = make_float2(fmaf(f, a.x, o0.x), fmaf(f, a.y, o0.y));
            o1 = make_float2(fmaf(f, c.x, o1.x), fmaf(f, c.y, o1.y));
        };
        if (pb[0] != -INFINITY) {
            const float f = exp2f(pb[0] - M);
            if (lane == 0) L = f * pb[1];
            add(pb, f);
        }
        for (int i0 = 0; i0 < n; i0 += 32) {
            // lane i: the weight of partial w0 + i0 + i (0 if it does not exist) and its share of L
            const int wi = w0 + i0 + lane;
            float f = 0.f;
            if (i0 + lane < n && owns(wi)) {
                const float* ph = slot(wi);
                f = exp2f(ph[0] - M);
                L = fmaf(f, ph[1], L);
            }
            const int m = min(32, n - i0);
            int k = 0;
            for (; k + 4 <= m; k += 4) {
                float fk[4];
                float2 a[4], c[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    fk[e] = __shfl_sync(0xffffffffu, f, k + e);
                    const float* ph = slot(w0 + i0 + k + e);
                    a[e] = fk[e] != 0.f ? *reinterpret_cast<const float2*>(ph + 2 + 2 * lane) : make_float2(0.f, 0.f);
                    c[e] = fk[e] != 0.f ? *reinterpret_cast<const float2*>(ph + 2 + 64 + 2 * lane) : make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    o0 = make_float2(fmaf(fk[e], a[e].x, o0.x), fmaf(fk[e], a[e].y, o0.y));
                    o1 = make_float2(fmaf(fk[e], c[e].x, o1.x), fmaf(fk[e], c[e].y, o1.y));
                }
            }
            for (; k < m; ++k) {
                const float fk = __shfl_sync(0xffffffffu, f, k);
                if (fk != 0.f) add(slot(w0 + i0 + k), fk);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        const float inv = 1.f / L;
        r0 = make_float2(o0.x * inv, o0.y * inv);
        r1 = make_float2(o1.x * inv, o1.y * inv);
    }
    // output row of head row hh: query token hh / g_real of the slot, head h * g_real + hh % g_real
    const int j = hh / p.g_real;
    if (j >= p.nq[b]) return;
    const size_t obase = (((size_t)p.q0[b] + j) * p.hkv * p.g_real + (size_t)h * p.g_real + hh % p.g_real) * kD;
    if (p.out_dtype == 0) {
        float* out = reinterpret_cast<float*>(p.out) + obase;
        *reinterpret_cast<float2*>(out + 2 * lane) = r0;
        *reinterpret_cast<float2*>(out + 64 + 2 * lane) = r1;
    } else {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + obase;
        *reinterpret_cast<__nv_bfloat162*>(out + 2 * lane) = __floats2bfloat162_rn(r0.x, r0.y);
        *reinterpret_cast<__nv_bfloat162*>(out + 64 + 2 * lane) = __floats2bfloat162_rn(r1.x, r1.y);
    }
}

template <int G>
cudaError_t launch_split(const DecodeParams& p, int max_ns, cudaStream_t s) {
    split_simt<G><<<dim3(max_ns, p.hkv, p.batch), 128, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const DecodeParams& p, const AppendParams& a, cudaStream_t s, cudaEvent_t* timing) {
    static_assert(sizeof(DecodeParams) + sizeof(AppendParams) <= 32000, "kernel parameters of prep_step");
    if (p.path != 2) return cudaErrorInvalidValue;
    cudaError_t e = launch_prep_step(p, a, s);
    if (e != cudaSuccess) return e;
    count_launches(1);
    if (timing && (e = cudaEventRecord(timing[0], s)) != cudaSuccess) return e;
    e = launch_decode_mma(p, s);
    if (e != cudaSuccess) return e;
    if (timing && (e = cudaEventRecord(timing[1], s)) != cudaSuccess) return e;
    combine_mma<<<dim3(p.hkv, p.batch), 32 * p.g, 0, s>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s, cudaEvent_t* timing) {
    cudaError_t e;
    if (p.path == 2) {
        // warp-MMA path: prep (q rotation + BF16 part) -> INT2 attention -> combine
        e = launch_prep(p, s);
        if (e != cudaSuccess) return e;
        count_launches(1);
        if (timing && (e = cudaEventRecord(timing[0], s)) != cudaSuccess) return e;
        e = launch_decode_mma(p, s);
        if (e != cudaSuccess) return e;
        if (timing && (e = cudaEventRecord(timing[1], s)) != cudaSuccess) return e;
    } else {
        // SIMT path: q rotation -> INT2 splits + BF16 split -> combine
        int max_ns = 1;
        for (int b = 0; b < p.batch; ++b) max_ns = max(max_ns, int2_splits(p.len[b], p.pps) + 1);
        rotate_q<<<dim3(p.hkv, p.batch), 128, 0, s>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (timing && (e = cudaEventRecord(timing[0], s)) != cudaSuccess) return e;
        switch (p.g) {
            case 1: e = launch_split<1>(p, max_ns, s); break;
            case 2: e = launch_split<2>(p, max_ns, s); break;
            case 3: e = launch_split<3>(p, max_ns, s); break;
            case 4: e = launch_split<4>(p, max_ns, s); break;
            case 5: e = launch_split<5>(p, max_ns, s); break;
            case 6: e = launch_split<6>(p, max_ns, s); break;
            case 7: e = launch_split<7>(p, max_ns, s); break;
            case 8: e = launch_split<8>(p, max_ns, s); break;
            case 12: e = launch_split<12>(p, max_ns, s); break;
            case 16: e = launch_split<16>(p, max_ns, s); break;
            default: return cudaErrorInvalidValue;
        }
        if (e != cudaSuccess) return e;
        if (timing && (e = cudaEventRecord(timing[1], s)) != cudaSuccess) return e;
        count_launches(2);
    }
    if (p.path == 2)
        combine_mma<<<dim3(p.hkv, p.batch), 32 * p.g, 0, s>>>(p);
    else
        combine<<<dim3(p.hkv * p.g, p.batch), 128, 0, s>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace oscar
