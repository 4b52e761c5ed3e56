// decode_mma.cu -- fused paged GQA decode attention over INT2 pages, warp-level tensor-core MMAs.
//
// The read path of the axbrief.com OSCAR page, section "attention-statistics rotation +
// Triton kernels": keys and values are unpacked and dequantised on chip inside the attention
// pass, with nothing dequantised written back; the key rotation is applied to the query
// (q~ = q . R_K from rotate_q), which equals inverse-rotating every key (R_K orthogonal).
//
// Every warp works alone on a contiguous range of 64-token INT2 pages of the flattened
// (request, KV head, page) list, so all warps stream the same number of bytes whatever the
// request lengths.  A warp keeps its own ring of shared-memory stages filled by bulk-async
// copies (page-table entries fetched 32 pages ahead).  Per page it converts the fp16 per-token
// scales and minima once into an fp32 table in shared memory, then runs 32-token chunks (16 for
// G > 8); every page but the last of a request takes a copy of the chunk loop without tail checks
// in which the output MMAs of chunk c - 1 follow the score MMAs of chunk c, so that the chunks of a
// page form straight-line blocks the compiler can interleave.  Per chunk:
//   scores   S = Q~ K^T on mma.sync.m16n8k16 (fp16 in, fp32 accumulate): A = the query,
//            rows = head (fp16 high part) and head + 8 (fp16 low part, the rounding residue),
//            so S_hi + S_lo carries ~22 bits of q~; B = 2-bit key codes.  The page stores the
//            codes in fragment order (k_code_byte), so a thread's codes for one token arrive
//            in one 8-byte load, and each B register is one AND of a code word (or of the word
//            shifted right by 8) with 0x00030003 << 2r: two fp16 subnormals code * 4^r * 2^-24,
//            exact.  The 4^r of k-step ks (r = ks mod 4) is taken out of the query side
//            (A = q~ * 2^(6 - 2r)), and the query of each (request, KV head) is scaled by a power
//            of two so that its largest high part sits in [2^13, 2^14).  One accumulator per
//            64-channel group because each group has its own scale:
//            logit = 2^18 s_g S_g / qscale + m_g sum_{c in g} q~_c (log2 units);
//   softmax  online, per head, with a lazily raised reference max (output rescaled only when a
//            logit passes the reference by 2^tau, tested per thread first, so the row-group max
//            reduction runs only on that rare path; tau is set per (request, KV head) from the largest
//            value scale the write path recorded, so that P' stays inside fp16); logits are formed
//            relative to the reference and all the per-token arithmetic runs on packed fp32 pairs
//            (f32x2 FMA / MUL / ADD:
//            the two tokens 2 tig, 2 tig + 1 of a score column pair), which halves the FP32
//            instructions and, unlike scalar FFMA, overlaps the MMAs almost fully;
//   output   O^T += V^T P'^T on the same MMA: A = the value codes (rows = 16 channels), again
//            one AND per register from a 16-byte load in fragment order (v_code_byte), with
//            channel tile cm carrying 4^(cm mod 4) * 2^-24 (removed when the partial is
//            written); B = P' = p * s_V (fp16, columns = 8 heads) straight from the score
//            accumulators' register layout.  Centred values: one more MMA per k-step sums the
//            same fp16 P' (A = those P' registers; B = ones that pick the value group), and after
//            each page the output takes -1.5 times that sum, so it accumulates P' (code - 1.5), a
//            zero-mean factor that keeps the rounding of P' from adding up over long nearly flat
//            attention; the minimum term sum_t p (m_V + 1.5 s_V) runs on the CUDA cores.
// Tokens are in natural order everywhere: n-tile nt of a chunk holds tokens 8 nt .. 8 nt + 7,
// and PV k-step kk takes n-tiles 2 kk (k 0..7) and 2 kk + 1 (k 8..15).  At the end of each
// (request, KV head) run the warp writes (reference max, sum, unnormalised output) to the
// split-K partial buffer.
//
// Head counts whose query rows would leave MMA rows empty (G <= 4, G = 12) run the transposed-score
// kernel of decode_mma_t.cu instead.
//
// mbarrier waits are bounded; on timeout the kernel records an error word and the warp stops.
#include <cuda_fp16.h>

#include "decode_mma_common.h"

namespace oscar {
namespace {

using namespace ptx;
using namespace mma_common;

// warps per CTA: 12 (168 registers each) when one m-tile holds the G heads (G <= 8); 8 (255
// registers) for two head tiles, whose query fragments and accumulators need twice the registers
__host__ __device__ constexpr int warps_for(int G) { return G <= 8 ? 12 : 8; }
// page stages per warp: 2 for one head tile (measured: no slower than 3, and 61 KB of shared memory
// freed), 3 for two head tiles, whose longer compute per page needs the deeper prefetch
__host__ __device__ constexpr int stages_for(int G) { return G <= 8 ? 2 : 3; }
template <int W, int S>
struct MmaSmem {
    uint8_t stage[W][S][kPageHeadBytes];
    uint64_t full[W][S];
    // per-token scales of the current page, token pairs (2p, 2p + 1) side by side:
    // [0] key (2^18 s0, 2^18 s0'), (m0, m0'); [1] key (2^18 s1, ...), (m1, ...); [2] value (s0, ...), (m0, ...);
    // [3] value (s1, ...), (m1, ...)
    float4 tsc[W][4][32];
    float tau[W];       // each warp's reference slack tau (log2 units), see the kernel
};


// FMT64: the default page format (keys and values in groups of 64) as compile-time offsets;
// otherwise the cache's format is read from the parameters.
template <int G, bool FMT64>
__global__ void __launch_bounds__(32 * warps_for(G), 1) decode_mma(const __grid_constant__ DecodeParams p) {
    constexpr int MT = (G + 7) / 8;              // heads per thread (rows g and g + 8 of each m-tile)
    constexpr int NT = MT == 1 ? 4 : 2;          // score n-tiles per chunk (8 tokens each)
    constexpr int CT = 8 * NT;                   // tokens per chunk
    constexpr int KK = NT / 2;                   // PV k-steps per chunk
    extern __shared__ __align__(128) uint8_t smem_raw[];
    constexpr int W = warps_for(G);
    constexpr int kStagesPerWarp = stages_for(G);
    MmaSmem<W, kStagesPerWarp>* sm = reinterpret_cast<MmaSmem<W, kStagesPerWarp>*>(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const PageFmt f = FMT64 ? page_fmt(64, 64) : p.fmt;
    const int gw = blockIdx.x * W + warp;
    const int P0 = (int)(((long long)gw * p.total_pages) / p.n_units);
    const int P1 = (int)(((long long)(gw + 1) * p.total_pages) / p.n_units);
    const int n = P1 - P0;
    if (lane == 0) {
        for (int s = 0; s < kStagesPerWarp; ++s) mbar_init(smem_u32(&sm->full[warp][s]), 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (n <= 0) return;

    // ---- page-table prefetch: lane l holds the pool block (physical page * hkv + KV head) of page
    // (base + l)
    auto fetch_pt = [&](int base) -> int32_t {
        const int P = P0 + base + lane;
        if (base + lane >= n) return 0;
        PageIt t;
        t.init(p, P);
        return p.page_table[(size_t)p.row[t.b] * p.max_pps + t.j] * p.hkv + t.h;
    };
    int pt_base = 0;
    int32_t pt_cur = fetch_pt(0);
    int32_t pt_nxt = fetch_pt(32);
    int issued = 0;
    auto issue = [&]() {   // lane 0: copy page `issued` into its stage
        const int q = issued;
        const int32_t blk = __shfl_sync(0xffffffffu, (q - pt_base) < 32 ? pt_cur : pt_nxt, (q - pt_base) & 31);
        if (lane == 0) {
            const int s = q % kStagesPerWarp;
            const uint32_t bar = smem_u32(&sm->full[warp][s]);
            mbar_expect_tx(bar, f.bytes);
            bulk_g2s(smem_u32(sm->stage[warp][s]), p.pool + (size_t)blk * f.bytes, f.bytes, bar);
        }
        ++issued;
    };
    for (int k = 0; k < kStagesPerWarp && k < n; ++k) issue();

    // ---- per-segment state
    uint32_t qa[MT][8][4];          // query fragments (hi rows g, lo rows g + 8) per head slot and k-step
    float qs[MT][2];                // sum over each channel group of (q_hi + q_lo)
    float mref[MT];
    float2 lsum[MT], mv[MT][2];     // per token parity e, summed when the partial is written
    bool fresh = true;
    float qscale = 1.f, kscale = kTwo18;   // power-of-two query scale of the segment and 2^18 / it
    // Reference-max slack tau (log2 units): probabilities stay at most 2^tau, and tau is set so that
    // 2^tau times the largest value scale of the (request, KV head) stays below 2^15, so that
    // P' = p * s_V cannot overflow fp16.  A raise of the reference puts the largest logit at
    // tau - 7.5, so the dominant probabilities sit about 2^7.5 below the limit.  tau lives in shared
    // memory (sm->tau[warp]): it is set once per segment and read once per chunk.
    float o[8][MT][4];              // output^T accumulators: channel tile cm, head tile nh
    // sums of P' over the current page for this thread's head g (+ 8 k) and value group tig / 2:
    // [0] over the first 8 tokens of each k-step, [2] over the last 8 ([1], [3] repeat them)
    float psum[MT][4];
    PageIt it;
    it.init(p, P0);
    bool seg_start = true;

    int consumed = 0;
    for (int i = 0; i < n; ++i) {
        const int s = i % kStagesPerWarp;
        if (seg_start) {
            // power-of-two query scale of this (request, KV head): the largest |q~| of its G heads,
            // times log2(e) / sqrt(128) * 2^6, lands in [2^13, 2^14), so the fp16 high parts cannot
            // overflow and keep 11 significant bits whatever the query's magnitude.  It is exact and
            // taken out again through the key-scale factor and the minimum sums (qs).
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < MT; ++k) {
                const int hd = g + 8 * k;
                const float* qr = p.qrot + (((size_t)it.b * p.hkv + it.h) * G + (hd < G ? hd : 0)) * kD;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const float2 q0 = *reinterpret_cast<const float2*>(qr + 16 * ks + 2 * tig);
                    const float2 q1 = *reinterpret_cast<const float2*>(qr + 16 * ks + 2 * tig + 8);
                    if (hd < G) amax = fmaxf(amax, fmaxf(fmaxf(fabsf(q0.x), fabsf(q0.y)), fmaxf(fabsf(q1.x), fabsf(q1.y))));
                }
            }
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
            {
                // floor(log2(amax * log2(e) / sqrt(128) * 64)) from the exponent field; the exponent
                // of the scale is clamped so that 2^e stays a normal fp32 number
                const int ex = (int)((__float_as_uint(amax * (kQScaleM * 64.f)) >> 23) & 0xff) - 127;
                const int e = max(-120, min(120, 13 - ex));
                qscale = __uint_as_float((uint32_t)(127 + e) << 23);
                kscale = __uint_as_float((uint32_t)(127 + 18 - e) << 23);    // 2^18 / qscale
            }
            const float qinv = __uint_as_float((uint32_t)(127 + 127 - ((__float_as_uint(qscale) >> 23) & 0xff)) << 23);
            // query fragments of this (request, KV head): k-step ks holds channels 16 ks + 2 tig + e
            // (+ 8 for registers 2, 3), scaled by 2^(6 - 2 (ks mod 4)) against the key codes' 4^r
#pragma unroll
            for (int k = 0; k < MT; ++k) {
                const int hd = g + 8 * k;
                float part0 = 0.f, part1 = 0.f;
                const float* qr = p.qrot + (((size_t)it.b * p.hkv + it.h) * G + (hd < G ? hd : 0)) * kD;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const float pw = (float)(64 >> (2 * (ks & 3)));      // 2^(6 - 2r), exact
                    const float sc = kQScaleM * pw * qscale, inv = qinv / pw;
                    const float2 q0 = *reinterpret_cast<const float2*>(qr + 16 * ks + 2 * tig);
                    const float2 q1 = *reinterpret_cast<const float2*>(qr + 16 * ks + 2 * tig + 8);
                    const float qv[2][2] = {{q0.x, q0.y}, {q1.x, q1.y}};
                    float hv[2][2], lv[2][2];
#pragma unroll
                    for (int f = 0; f < 2; ++f)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float q = hd < G ? qv[f][e] * sc : 0.f;
                            const float h = __half2float(__float2half_rn(q));
                            const float l = __half2float(__float2half_rn(q - h));
                            hv[f][e] = h;
                            lv[f][e] = l;
                            if (ks < 4) part0 += (h + l) * inv;
                            else part1 += (h + l) * inv;
                        }
                    qa[k][ks][0] = pack_h2(hv[0][0], hv[0][1]);
                    qa[k][ks][1] = pack_h2(lv[0][0], lv[0][1]);
                    qa[k][ks][2] = pack_h2(hv[1][0], hv[1][1]);
                    qa[k][ks][3] = pack_h2(lv[1][0], lv[1][1]);
                }
                part0 += __shfl_xor_sync(0xffffffffu, part0, 1);
                part0 += __shfl_xor_sync(0xffffffffu, part0, 2);
                part1 += __shfl_xor_sync(0xffffffffu, part1, 1);
                part1 += __shfl_xor_sync(0xffffffffu, part1, 2);
                qs[k][0] = part0;
                qs[k][1] = part1;
                mref[k] = 0.f;
                lsum[k] = mv[k][0] = mv[k][1] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
#pragma unroll
                for (int k = 0; k < MT; ++k) o[c][k][0] = o[c][k][1] = o[c][k][2] = o[c][k][3] = 0.f;
#pragma unroll
            for (int k = 0; k < MT; ++k) psum[k][0] = psum[k][1] = psum[k][2] = psum[k][3] = 0.f;
            seg_start = false;
            fresh = true;
            if (lane == 0) {
                // tau from the largest value scale the write path has quantised for this (request,
                // KV head): 2^tau * s_V in [2^14, 2^15) for the largest s_V, so P' = p * s_V < 2^15
                const uint32_t w16 = p.vmax[(size_t)p.row[it.b] * p.hkv + it.h] & 0xffffu;
                float tau = kTauMax;
                if (w16) {
                    const float w = __half2float(__ushort_as_half((unsigned short)w16));
                    tau = fminf(kTauMax, (float)(14 - ((int)((__float_as_uint(w) >> 23) & 0xff) - 127)));
                }
                sm->tau[warp] = tau;
            }
            __syncwarp();
        }
        const bool got = wait_full(smem_u32(&sm->full[warp][s]), (i / kStagesPerWarp) & 1, p.err, p.wait_iters);
        if (!__all_sync(0xffffffffu, got)) break;      // error word set; stop issuing, drain below
        consumed = i + 1;
        const uint8_t* pg = sm->stage[warp][s];
        const int n_live = min(kPage, int2_tokens(p.len[it.b]) - it.j * kPage);

        // ---- per-token scales of the page (tokens lane and lane + 32), staged in shared memory;
        // the warp barrier before the stage refill orders the previous page's reads before these writes.
        // Slots past the request's end are staged as 0 (their bytes may be anything); a full page
        // takes a copy of the loop without that test
        auto stage = [&](const bool full) {
        // thread = token pair (2 lane, 2 lane + 1): its scales and minima are one 16-byte load per
        // tensor (8 bytes for 128-channel groups), its four table entries one 16-byte store each
        const int t0 = 2 * lane;
        const bool live0 = full || t0 < n_live, live1 = full || t0 + 1 < n_live;
        uint4 ksm, vsm;   // (s, m) of group 0 / 1 for token t0 (x, y) and t0 + 1 (z, w)
        if (FMT64 || f.gk == 64) {
            ksm = *reinterpret_cast<const uint4*>(pg + kKSm + t0 * 8);
        } else {   // one (s, m) pair per token for both halves of a 128-channel group
            const uint2 k2 = *reinterpret_cast<const uint2*>(pg + kKSm + t0 * 4);
            ksm = make_uint4(k2.x, k2.x, k2.y, k2.y);
        }
        if (FMT64 || f.gv == 64) {
            vsm = *reinterpret_cast<const uint4*>(pg + f.v_sm + t0 * 8);
        } else {
            const uint2 v2 = *reinterpret_cast<const uint2*>(pg + f.v_sm + t0 * 4);
            vsm = make_uint4(v2.x, v2.x, v2.y, v2.y);
        }
        auto lo = [](uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffff))); };
        auto hi = [](uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); };
        // keys: (2^18 / qscale) s and m; values: s and the centred minimum m + 1.5 s (the output MMAs
        // take code - 1.5).  Slots past the request's end are staged as 0
        const float sv00 = live0 ? lo(vsm.x) : 0.f, sv01 = live0 ? lo(vsm.y) : 0.f;
        const float sv10 = live1 ? lo(vsm.z) : 0.f, sv11 = live1 ? lo(vsm.w) : 0.f;
        float4* row = &sm->tsc[warp][0][lane];
        row[0] = make_float4(live0 ? kscale * lo(ksm.x) : 0.f, live1 ? kscale * lo(ksm.z) : 0.f,
                             live0 ? hi(ksm.x) : 0.f, live1 ? hi(ksm.z) : 0.f);
        row[32] = make_float4(live0 ? kscale * lo(ksm.y) : 0.f, live1 ? kscale * lo(ksm.w) : 0.f,
                              live0 ? hi(ksm.y) : 0.f, live1 ? hi(ksm.w) : 0.f);
        row[64] = make_float4(sv00, sv10, live0 ? fmaf(1.5f, sv00, hi(vsm.x)) : 0.f,
                              live1 ? fmaf(1.5f, sv10, hi(vsm.z)) : 0.f);
        row[96] = make_float4(sv01, sv11, live0 ? fmaf(1.5f, sv01, hi(vsm.y)) : 0.f,
                              live1 ? fmaf(1.5f, sv11, hi(vsm.w)) : 0.f);
        };
        if (n_live == kPage) stage(true);
        else stage(false);
        __syncwarp();

        // scores and logits of one chunk, relative to the current reference max
        auto scores = [&](const int cbase, const bool partial, float2 (&lg)[MT][NT]) {
            // ---- scores: acc[k][nt][group]; n-tile nt = tokens cbase + 8 nt + (0..7)
            float acc[MT][NT][2][4];
#pragma unroll
            for (int k = 0; k < MT; ++k)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int gr = 0; gr < 2; ++gr) acc[k][nt][gr][0] = acc[k][nt][gr][1] = acc[k][nt][gr][2] = acc[k][nt][gr][3] = 0.f;
            {
                // this thread's 32 codes of token cbase + 8 nt + g: word u = channel group u
                uint32_t wl[NT][2], wh[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint2 kw = *reinterpret_cast<const uint2*>(pg + kKCodes + (cbase + 8 * nt + g) * 32 + 8 * tig);
                    wl[nt][0] = kw.x;
                    wl[nt][1] = kw.y;
                    wh[nt][0] = kw.x >> 8;
                    wh[nt][1] = kw.y >> 8;
                }
                // k-step 4u + R of every n-tile; consecutive MMAs go to different accumulators
#define OSCAR_QK_STEP(R)                                                                                    \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) _Pragma("unroll") for (int u = 0; u < 2; ++u) {      \
        const uint32_t b0 = code_pair<R>(wl[nt][u]), b1 = code_pair<R>(wh[nt][u]);                          \
        _Pragma("unroll") for (int k = 0; k < MT; ++k) mma16816(acc[k][nt][u], qa[k][4 * u + R], b0, b1);  \
    }
                OSCAR_QK_STEP(0)
                OSCAR_QK_STEP(1)
                OSCAR_QK_STEP(2)
                OSCAR_QK_STEP(3)
#undef OSCAR_QK_STEP
            }

            // ---- logits (packed over the token pair e = 0, 1 of each n-tile column pair), relative
            // to the reference max
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float4 k0 = sm->tsc[warp][0][(cbase >> 1) + 4 * nt + tig], k1 = sm->tsc[warp][1][(cbase >> 1) + 4 * nt + tig];
#pragma unroll
                for (int k = 0; k < MT; ++k) {
                    const float2 s0 = __fadd2_rn(make_float2(acc[k][nt][0][0], acc[k][nt][0][1]),
                                                 make_float2(acc[k][nt][0][2], acc[k][nt][0][3]));
                    const float2 s1 = __fadd2_rn(make_float2(acc[k][nt][1][0], acc[k][nt][1][1]),
                                                 make_float2(acc[k][nt][1][2], acc[k][nt][1][3]));
                    float2 x = __ffma2_rn(make_float2(k1.z, k1.w), make_float2(qs[k][1], qs[k][1]),
                                          make_float2(-mref[k], -mref[k]));
                    x = __ffma2_rn(make_float2(k0.z, k0.w), make_float2(qs[k][0], qs[k][0]), x);
                    x = __ffma2_rn(make_float2(k1.x, k1.y), s1, x);
                    lg[k][nt] = __ffma2_rn(make_float2(k0.x, k0.y), s0, x);
                }
            }
            if (partial) {
                // tokens past the request's end: probability 0 (their scales were staged as 0)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
#pragma unroll
                        for (int k = 0; k < MT; ++k)
                            if (cbase + 8 * nt + 2 * tig + e >= n_live) (e ? lg[k][nt].y : lg[k][nt].x) = -INFINITY;
            }
        };
        // reference-max update (thread-local test, rare warp-wide raise)
        auto update = [&](float2 (&lg)[MT][NT]) {
            const float tau = sm->tau[warp];
            // thread-local test first: the row-group reduction runs only when some logit of the
            // warp passed the reference by 2^tau (or the segment is fresh)
            float cml[MT];
            bool hot = fresh;
#pragma unroll
            for (int k = 0; k < MT; ++k) {
                float cm = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) cm = fmaxf(cm, fmaxf(lg[k][nt].x, lg[k][nt].y));
                cml[k] = cm;
                hot = hot || cm > tau;
            }
            if (__any_sync(0xffffffffu, hot)) {
                float fown[MT], cmx[MT];
#pragma unroll
                for (int k = 0; k < MT; ++k) {
                    float cm = cml[k];
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
                    fown[k] = 1.f;
                    cmx[k] = 0.f;
                    if (fresh || cm > tau) {
                        // the reference rises so that the largest logit sits at tau - 7.5
                        const float d = cm - (tau - kTauSlack);
                        fown[k] = fresh ? 0.f : ex2(-d);
                        mref[k] += d;
                        cmx[k] = d;
                        const float2 f2 = make_float2(fown[k], fown[k]);
                        lsum[k] = __fmul2_rn(lsum[k], f2);
                        mv[k][0] = __fmul2_rn(mv[k][0], f2);
                        mv[k][1] = __fmul2_rn(mv[k][1], f2);
                        psum[k][0] *= fown[k];
                        psum[k][1] *= fown[k];
                        psum[k][2] *= fown[k];
                        psum[k][3] *= fown[k];
                    }
                }
                fresh = false;
#pragma unroll
                for (int k = 0; k < MT; ++k)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) lg[k][nt] = __fadd2_rn(lg[k][nt], make_float2(-cmx[k], -cmx[k]));
                // a head's reference max went up; O^T holds heads 2 tig, 2 tig + 1 (+ 8 nh),
                // whose factors live in the threads of rows g = head
#pragma unroll
                for (int k = 0; k < MT; ++k) {
                    const float f0 = __shfl_sync(0xffffffffu, fown[k], (2 * tig) * 4);
                    const float f1 = __shfl_sync(0xffffffffu, fown[k], (2 * tig + 1) * 4);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        o[c][k][0] *= f0;
                        o[c][k][1] *= f1;
                        o[c][k][2] *= f0;
                        o[c][k][3] *= f1;
                    }
                }
            }
        };
        // probabilities and P' of one chunk
        auto probs = [&](const int cbase, const float2 (&lg)[MT][NT], uint32_t (&pb)[2][KK][MT][2]) {
            // probabilities (ex2(-inf) = 0) and P' = p * s_V rounded once to fp16, packed per token pair
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float4 v0 = sm->tsc[warp][2][(cbase >> 1) + 4 * nt + tig], v1 = sm->tsc[warp][3][(cbase >> 1) + 4 * nt + tig];
                const int kk = nt >> 1, half = nt & 1;
#pragma unroll
                for (int k = 0; k < MT; ++k) {
                    const float2 pr = make_float2(ex2(lg[k][nt].x), ex2(lg[k][nt].y));
                    lsum[k] = __fadd2_rn(lsum[k], pr);
                    mv[k][0] = __ffma2_rn(pr, make_float2(v0.z, v0.w), mv[k][0]);
                    mv[k][1] = __ffma2_rn(pr, make_float2(v1.z, v1.w), mv[k][1]);
                    const float2 p0 = __fmul2_rn(pr, make_float2(v0.x, v0.y));
                    const float2 p1 = __fmul2_rn(pr, make_float2(v1.x, v1.y));
                    pb[0][kk][k][half] = pack_h2(p0.x, p0.y);
                    pb[1][kk][k][half] = pack_h2(p1.x, p1.y);
                }
            }

        };
        // O^T += V^T P'^T of one chunk
        auto pv = [&](const int cbase, const uint32_t (&pb)[2][KK][MT][2]) {
            // ---- output^T: O[cm] += V^T[channels 16 cm + g, + 8][tokens] x P'_{group(cm)}
            // value words of this thread for the chunk's k-steps: [channel half q][k-step][s]
            {
                const uint8_t* vsrc = pg + f.v_codes + 1024 * (cbase >> 5) + 16 * lane;
                uint32_t vw[2][KK][2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    if constexpr (KK == 2) {
                        const uint4 w4 = *reinterpret_cast<const uint4*>(vsrc + 512 * q);
                        vw[q][0][0] = w4.x;
                        vw[q][0][1] = w4.y;
                        vw[q][1][0] = w4.z;
                        vw[q][1][1] = w4.w;
                    } else {
                        const uint2 w2 = *reinterpret_cast<const uint2*>(vsrc + 512 * q + 8 * ((cbase >> 4) & 1));
                        vw[q][0][0] = w2.x;
                        vw[q][0][1] = w2.y;
                    }
                }
                // k-step outer: the MMAs into one accumulator are 8 apart
#pragma unroll
                for (int kk = 0; kk < KK; ++kk)
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        const uint32_t w0 = vw[q][kk][0], w1 = vw[q][kk][1];
                        const uint32_t s0 = w0 >> 8, s1 = w1 >> 8;
#define OSCAR_PV_STEP(R)                                                                                 \
    {                                                                                                    \
        const uint32_t av[4] = {code_pair<R>(w0), code_pair<R>(s0), code_pair<R>(w1), code_pair<R>(s1)}; \
        _Pragma("unroll") for (int k = 0; k < MT; ++k)                                                   \
            mma16816(o[4 * q + R][k], av, pb[q][kk][k][0], pb[q][kk][k][1]);                             \
    }
                        OSCAR_PV_STEP(0)
                        OSCAR_PV_STEP(1)
                        OSCAR_PV_STEP(2)
                        OSCAR_PV_STEP(3)
#undef OSCAR_PV_STEP
                    }
                // the page's sums of P', of exactly the fp16 values the output MMAs see.  A = the
                // output MMAs' B registers of the k-step in their own order, so row g holds head g's
                // P' of tokens 0..7 (group 0 in k 0..7, group 1 in k 8..15) and row g + 8 those of
                // tokens 8..15; B = 1 on (k 0..7, columns 0..3) and (k 8..15, columns 4..7).  Result
                // columns 0..3 then sum group 0 and columns 4..7 group 1, each over half the tokens
                // in rows g and g + 8
                const uint32_t sb0 = (g < 4) ? 0x3C003C00u : 0u, sb1 = (g < 4) ? 0u : 0x3C003C00u;
#pragma unroll
                for (int kk = 0; kk < KK; ++kk)
#pragma unroll
                    for (int k = 0; k < MT; ++k) {
                        const uint32_t pa[4] = {pb[0][kk][k][0], pb[0][kk][k][1], pb[1][kk][k][0], pb[1][kk][k][1]};
                        mma16816(psum[k], pa, sb0, sb1);
                    }
            }
        };
        constexpr int NC = kPage / CT;
        if (n_live == kPage) {   // every page but the last of a request: output MMAs of chunk c - 1 after the scores of chunk c
            float2 lg[MT][NT];
            uint32_t pbs[2][2][KK][MT][2];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                scores(c * CT, false, lg);
                if (c > 0) pv((c - 1) * CT, pbs[(c - 1) & 1]);
                update(lg);
                probs(c * CT, lg, pbs[c & 1]);
            }
            pv((NC - 1) * CT, pbs[(NC - 1) & 1]);
        } else {
#pragma unroll
            for (int cbase = 0; cbase < kPage; cbase += CT) {
                if (cbase >= n_live) break;
                float2 lg[MT][NT];
                uint32_t pb[2][KK][MT][2];
                scores(cbase, cbase + CT > n_live, lg);
                update(lg);
                probs(cbase, lg, pb);
                pv(cbase, pb);
            }
        }

        // ---- centre the page's output: -1.5 P' per head and value group, in the units of channel
        // tile cm (4^(cm mod 4) 2^-24), then start the next page's sum.  O^T holds heads 2 tig,
        // 2 tig + 1 (+ 8 k); the sum of head h's group q sits in lane 4 h + 2 q
        float ps_a[MT][2], ps_b[MT][2];
#pragma unroll
        for (int k = 0; k < MT; ++k) {
            const float t = psum[k][0] + psum[k][2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                ps_a[k][q] = __shfl_sync(0xffffffffu, t, (2 * tig) * 4 + 2 * q);
                ps_b[k][q] = __shfl_sync(0xffffffffu, t, (2 * tig + 1) * 4 + 2 * q);
            }
        }
#pragma unroll
        for (int cm = 0; cm < 8; ++cm) {
            const float c = -1.5f * (float)(1 << (2 * (cm & 3))) * 5.9604644775390625e-08f;   // -1.5 * 4^r * 2^-24
            const int q = cm >> 2;
#pragma unroll
            for (int k = 0; k < MT; ++k) {
                const float2 sq = make_float2(ps_a[k][q], ps_b[k][q]);
                const float2 cc = make_float2(c, c);
                const float2 a = __ffma2_rn(cc, sq, make_float2(o[cm][k][0], o[cm][k][1]));
                const float2 b = __ffma2_rn(cc, sq, make_float2(o[cm][k][2], o[cm][k][3]));
                o[cm][k][0] = a.x;
                o[cm][k][1] = a.y;
                o[cm][k][2] = b.x;
                o[cm][k][3] = b.y;
            }
        }
#pragma unroll
        for (int k = 0; k < MT; ++k) psum[k][0] = psum[k][1] = psum[k][2] = psum[k][3] = 0.f;

        // ---- stage consumed: refill it with the page kStagesPerWarp ahead
        __syncwarp();
        fence_proxy_async();
        if (issued < n) {
            if (issued >= pt_base + 32) {
                pt_base += 32;
                pt_cur = pt_nxt;
                pt_nxt = fetch_pt(pt_base + 32);
            }
            issue();
        }

        // ---- end of this warp's part of a (request, KV head) run: write the partial result
        const bool last = (i == n - 1);
        const int b_now = it.b, h_now = it.h;
        const bool new_seg = it.next(p);
        if (last || new_seg) {
            float* part = p.part_mma + ((size_t)(b_now * p.hkv + h_now) + gw) * G * (2 + kD);
#pragma unroll
            for (int k = 0; k < MT; ++k) {
                // per-head totals over the four threads of the head's row group
                float l = lsum[k].x + lsum[k].y, m0 = mv[k][0].x + mv[k][0].y, m1 = mv[k][1].x + mv[k][1].y;
                l += __shfl_xor_sync(0xffffffffu, l, 1);
                l += __shfl_xor_sync(0xffffffffu, l, 2);
                m0 += __shfl_xor_sync(0xffffffffu, m0, 1);
                m0 += __shfl_xor_sync(0xffffffffu, m0, 2);
                m1 += __shfl_xor_sync(0xffffffffu, m1, 1);
                m1 += __shfl_xor_sync(0xffffffffu, m1, 2);
                const int hown = g + 8 * k;
                if (hown < G && tig == 0) {
                    part[(size_t)hown * (2 + kD) + 0] = mref[k];
                    part[(size_t)hown * (2 + kD) + 1] = l;
                }
                // this thread's output entries: heads 8 k + 2 tig + e, channels 16 cm + g (+ 8)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int hd = 8 * k + 2 * tig + e;
                    const float mh0 = __shfl_sync(0xffffffffu, m0, (2 * tig + e) * 4);
                    const float mh1 = __shfl_sync(0xffffffffu, m1, (2 * tig + e) * 4);
                    if (hd < G) {
                        float* ph = part + (size_t)hd * (2 + kD) + 2;
#pragma unroll
                        for (int cm = 0; cm < 8; ++cm) {
                            // channel tile cm was accumulated at 4^(cm mod 4) * 2^-24 per code
                            const float sc = (float)(1 << (24 - 2 * (cm & 3)));
                            const float mg = cm < 4 ? mh0 : mh1;
                            ph[16 * cm + g] = fmaf(sc, o[cm][k][e], mg);
                            ph[16 * cm + g + 8] = fmaf(sc, o[cm][k][2 + e], mg);
                        }
                    }
                }
            }
            seg_start = true;
        }
    }
    // copies still in flight must land before the warp may exit (only after a timeout)
    if (lane == 0)
        for (int q = consumed; q < issued; ++q)
            wait_full(smem_u32(&sm->full[warp][q % kStagesPerWarp]), (q / kStagesPerWarp) & 1, p.err, kDrainIters);
}

template <int G, bool FMT64>
cudaError_t launch_mma_gf(const DecodeParams& p, cudaStream_t s) {
    constexpr int W = warps_for(G);
    const int smem = (int)sizeof(MmaSmem<W, stages_for(G)>);
    static bool attr_set[kMaxDevices] = {};   // once per instantiation and device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(decode_mma<G, FMT64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    decode_mma<G, FMT64><<<p.n_units / W, 32 * W, smem, s>>>(p);
    return cudaGetLastError();
}

template <int G>
cudaError_t launch_mma_g(const DecodeParams& p, cudaStream_t s) {
    if (p.fmt.gk == 64 && p.fmt.gv == 64) return launch_mma_gf<G, true>(p, s);
    return launch_mma_gf<G, false>(p, s);
}

}  // namespace

int mma_units_per_cta(int g) { return decode_mma_t_serves(g) ? mma_t_units_per_cta(g) : warps_for(g); }

cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t s) {
    if (p.total_pages == 0) return cudaSuccess;
    count_launches(1);
    if (decode_mma_t_serves(p.g)) return launch_decode_mma_t(p, s);   // query rows would leave MMA rows empty
    switch (p.g) {
        case 5: return launch_mma_g<5>(p, s);
        case 6: return launch_mma_g<6>(p, s);
        case 7: return launch_mma_g<7>(p, s);
        case 8: return launch_mma_g<8>(p, s);
        case 12: return launch_mma_g<12>(p, s);
        case 16: return launch_mma_g<16>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace oscar
