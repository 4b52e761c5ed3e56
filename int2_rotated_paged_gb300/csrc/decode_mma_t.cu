// decode_mma_t.cu -- fused paged GQA decode attention over INT2 pages with the scores taken
// transposed: S^T = K Q~^T, the key codes as the warp MMA's A operand and the query as B.
//
// The read path of the axbrief.com OSCAR page, section "attention-statistics rotation + Triton
// kernels", as in decode_mma.cu, for the head counts where the query-as-A form leaves MMA rows
// empty.  There a 16-row query tile holds 8 heads (fp16 high part in rows g, low part in rows
// g + 8), so G <= 4 fills half of one tile and G = 12 three quarters of two.  Here the query is
// the 8-column B operand, 4 heads per n-tile with each head's high and low parts in adjacent
// columns, and A holds the codes of 16 tokens: G <= 4 takes one n-tile, half the score MMAs of the
// query-as-A form, and G = 12 three n-tiles, three quarters of them.  A's four registers are the
// code words decode_mma.cu feeds as B for two 8-token n-tiles, so the unpacking is the same.
//
// Each lane owns one head of every n-tile (head 4 j + tig) for the tokens g and g + 8 of every
// 16-token m-tile: the softmax runs on real heads only, its per-token work packed as (g, g + 8)
// pairs on f32x2 FMAs.  P' = p * s_V is packed per lane as the fp16 pair (token g, token g + 8)
// and moved into the output MMA's B layout (tokens 2 tig, 2 tig + 1 of head g) with two shuffles
// and one byte permute per register.  From there on (output MMAs O^T += V^T P'^T, the page sums of
// P', the centred values, the partial results) the kernel is decode_mma.cu's.
//
// mbarrier waits are bounded; on timeout the kernel records an error word and the warp stops.
#include "decode_mma_common.h"

namespace oscar {
namespace {

using namespace ptx;
using namespace mma_common;

// warps per CTA and page stages per warp, as for decode_mma.cu with the same output head tiles
__host__ __device__ constexpr int warps_t(int G) { return G <= 8 ? 12 : 8; }
__host__ __device__ constexpr int stages_t(int G) { return G <= 8 ? 2 : 3; }

template <int W, int S>
struct MmaTSmem {
    uint8_t stage[W][S][kPageHeadBytes];
    uint64_t full[W][S];
    // per-token scales of the current page by 16-token m-tile mt and row r, the tokens
    // t0 = 16 mt + r and t1 = t0 + 8 side by side: [0] key group 0 (2^18 s / qscale (t0, t1),
    // m (t0, t1)); [1] key group 1; [2] value group 0 (s (t0, t1), m + 1.5 s (t0, t1)); [3] value group 1
    float4 tsc[W][4][kPage / 16][8];
    float tau[W];       // each warp's reference slack tau (log2 units), see decode_mma.cu
};

// FMT64: the default page format (keys and values in groups of 64) as compile-time offsets;
// otherwise the cache's format is read from the parameters.
template <int G, bool FMT64>
__global__ void __launch_bounds__(32 * warps_t(G), 1) decode_mma_t(const __grid_constant__ DecodeParams p) {
    constexpr int NS = (G + 3) / 4;              // score n-tiles: 4 heads each, high and low parts side by side
    constexpr int MO = (G + 7) / 8;              // output head tiles of 8 heads
    constexpr int MK = G <= 4 ? 2 : 1;           // 16-token m-tiles per chunk
    constexpr int CT = 16 * MK;                  // tokens per chunk
    constexpr int KK = MK;                       // PV k-steps per chunk
    extern __shared__ __align__(128) uint8_t smem_raw[];
    constexpr int W = warps_t(G);
    constexpr int kStagesPerWarp = stages_t(G);
    MmaTSmem<W, kStagesPerWarp>* sm = reinterpret_cast<MmaTSmem<W, kStagesPerWarp>*>(smem_raw);
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
    uint32_t qb[NS][8][2];          // query B fragments of k-step ks: head 4 j + g / 2, high part (g even) or low
    float2 qs2[NS][2];              // (sum over channel group u of the used q~, the same) of head 4 j + tig
    float mref[NS];
    float2 nref[NS];                // (-mref, -mref)
    float2 lsum[NS], mv[NS][2];     // per token half (t0, t1), summed when the partial is written
    bool fresh = true;
    float qscale = 1.f, kscale = kTwo18;   // power-of-two query scale of the segment and 2^18 / it
    float o[8][MO][4];              // output^T accumulators: channel tile cm, head tile mo
    // sums of P' over the current page for head 8 mo + g and value group tig / 2: [0] over the
    // first 8 tokens of each k-step, [2] over the last 8 ([1], [3] repeat them)
    float psum[MO][4];
    PageIt it;
    it.init(p, P0);
    bool seg_start = true;

    int consumed = 0;
    for (int i = 0; i < n; ++i) {
        const int s = i % kStagesPerWarp;
        if (seg_start) {
            // power-of-two query scale of this (request, KV head), as in decode_mma.cu: the largest
            // |q~| of its G heads times log2(e) / sqrt(128) * 2^6 lands in [2^13, 2^14)
            const float* qbase = p.qrot + ((size_t)it.b * p.hkv + it.h) * G * kD;
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < NS; ++j) {
                const int hb = 4 * j + (g >> 1);
                const float* qr = qbase + (size_t)(hb < G ? hb : 0) * kD;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const float2 q0 = *reinterpret_cast<const float2*>(qr + 16 * ks + 2 * tig);
                    const float2 q1 = *reinterpret_cast<const float2*>(qr + 16 * ks + 2 * tig + 8);
                    if (hb < G) amax = fmaxf(amax, fmaxf(fmaxf(fabsf(q0.x), fabsf(q0.y)), fmaxf(fabsf(q1.x), fabsf(q1.y))));
                }
            }
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
            {
                const int ex = (int)((__float_as_uint(amax * (kQScaleM * 64.f)) >> 23) & 0xff) - 127;
                const int e = max(-120, min(120, 13 - ex));
                qscale = __uint_as_float((uint32_t)(127 + e) << 23);
                kscale = __uint_as_float((uint32_t)(127 + 18 - e) << 23);    // 2^18 / qscale
            }
            const float qinv = __uint_as_float((uint32_t)(127 + 127 - ((__float_as_uint(qscale) >> 23) & 0xff)) << 23);
            // query fragments: column g of n-tile j is head 4 j + g / 2, its fp16 high part for g even
            // and the rounding residue's fp16 for g odd; k-step ks holds channels 16 ks + 2 tig + e
            // (+ 8 for the second register), scaled by 2^(6 - 2 (ks mod 4)) against the codes' 4^r
#pragma unroll
            for (int j = 0; j < NS; ++j) {
                const int hb = 4 * j + (g >> 1);
                const bool low = g & 1;
                float part0 = 0.f, part1 = 0.f;
                const float* qr = qbase + (size_t)(hb < G ? hb : 0) * kD;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const float pw = (float)(64 >> (2 * (ks & 3)));      // 2^(6 - 2r), exact
                    const float sc = kQScaleM * pw * qscale, inv = qinv / pw;
                    const float2 q0 = *reinterpret_cast<const float2*>(qr + 16 * ks + 2 * tig);
                    const float2 q1 = *reinterpret_cast<const float2*>(qr + 16 * ks + 2 * tig + 8);
                    const float qv[2][2] = {{q0.x, q0.y}, {q1.x, q1.y}};
                    float v[2][2];
#pragma unroll
                    for (int fh = 0; fh < 2; ++fh)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float q = hb < G ? qv[fh][e] * sc : 0.f;
                            const float h = __half2float(__float2half_rn(q));
                            const float l = __half2float(__float2half_rn(q - h));
                            v[fh][e] = low ? l : h;
                            if (ks < 4) part0 += (h + l) * inv;
                            else part1 += (h + l) * inv;
                        }
                    qb[j][ks][0] = pack_h2(v[0][0], v[0][1]);
                    qb[j][ks][1] = pack_h2(v[1][0], v[1][1]);
                }
                // sums over the channels of the row group; head 4 j + tig's sit in row group 2 tig
                part0 += __shfl_xor_sync(0xffffffffu, part0, 1);
                part0 += __shfl_xor_sync(0xffffffffu, part0, 2);
                part1 += __shfl_xor_sync(0xffffffffu, part1, 1);
                part1 += __shfl_xor_sync(0xffffffffu, part1, 2);
                const float s0 = __shfl_sync(0xffffffffu, part0, (2 * tig) * 4);
                const float s1 = __shfl_sync(0xffffffffu, part1, (2 * tig) * 4);
                qs2[j][0] = make_float2(s0, s0);
                qs2[j][1] = make_float2(s1, s1);
                mref[j] = 0.f;
                nref[j] = make_float2(0.f, 0.f);
                lsum[j] = mv[j][0] = mv[j][1] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
#pragma unroll
                for (int k = 0; k < MO; ++k) o[c][k][0] = o[c][k][1] = o[c][k][2] = o[c][k][3] = 0.f;
#pragma unroll
            for (int k = 0; k < MO; ++k) psum[k][0] = psum[k][1] = psum[k][2] = psum[k][3] = 0.f;
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

        // ---- per-token scales of the page, staged in shared memory: lane = (m-tile lane / 8, row
        // lane % 8), its tokens t0 = 16 (lane / 8) + lane % 8 and t1 = t0 + 8, one 16-byte store per
        // table.  Slots past the request's end are staged as 0; the warp barrier before the stage
        // refill orders the previous page's reads before these writes
        auto stage = [&](const bool full) {
            const int mt = lane >> 3, r = lane & 7;
            const int t0 = 16 * mt + r, t1 = t0 + 8;
            const bool live0 = full || t0 < n_live, live1 = full || t1 < n_live;
            uint2 k0, k1, v0, v1;   // (s, m) of group 0 (x) and group 1 (y) of tokens t0, t1
            if (FMT64 || f.gk == 64) {
                k0 = *reinterpret_cast<const uint2*>(pg + kKSm + t0 * 8);
                k1 = *reinterpret_cast<const uint2*>(pg + kKSm + t1 * 8);
            } else {   // one (s, m) pair per token for both halves of a 128-channel group
                const uint32_t a = *reinterpret_cast<const uint32_t*>(pg + kKSm + t0 * 4);
                const uint32_t b = *reinterpret_cast<const uint32_t*>(pg + kKSm + t1 * 4);
                k0 = make_uint2(a, a);
                k1 = make_uint2(b, b);
            }
            if (FMT64 || f.gv == 64) {
                v0 = *reinterpret_cast<const uint2*>(pg + f.v_sm + t0 * 8);
                v1 = *reinterpret_cast<const uint2*>(pg + f.v_sm + t1 * 8);
            } else {
                const uint32_t a = *reinterpret_cast<const uint32_t*>(pg + f.v_sm + t0 * 4);
                const uint32_t b = *reinterpret_cast<const uint32_t*>(pg + f.v_sm + t1 * 4);
                v0 = make_uint2(a, a);
                v1 = make_uint2(b, b);
            }
            auto lo = [](uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffff))); };
            auto hi = [](uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); };
            const float sa0 = live0 ? lo(v0.x) : 0.f, sa1 = live0 ? lo(v0.y) : 0.f;
            const float sb0 = live1 ? lo(v1.x) : 0.f, sb1 = live1 ? lo(v1.y) : 0.f;
            sm->tsc[warp][0][mt][r] = make_float4(live0 ? kscale * lo(k0.x) : 0.f, live1 ? kscale * lo(k1.x) : 0.f,
                                                  live0 ? hi(k0.x) : 0.f, live1 ? hi(k1.x) : 0.f);
            sm->tsc[warp][1][mt][r] = make_float4(live0 ? kscale * lo(k0.y) : 0.f, live1 ? kscale * lo(k1.y) : 0.f,
                                                  live0 ? hi(k0.y) : 0.f, live1 ? hi(k1.y) : 0.f);
            sm->tsc[warp][2][mt][r] = make_float4(sa0, sb0, live0 ? fmaf(1.5f, sa0, hi(v0.x)) : 0.f,
                                                  live1 ? fmaf(1.5f, sb0, hi(v1.x)) : 0.f);
            sm->tsc[warp][3][mt][r] = make_float4(sa1, sb1, live0 ? fmaf(1.5f, sa1, hi(v0.y)) : 0.f,
                                                  live1 ? fmaf(1.5f, sb1, hi(v1.y)) : 0.f);
        };
        if (n_live == kPage) stage(true);
        else stage(false);
        __syncwarp();

        // scores and logits of one chunk, relative to the current reference max: lg[m][j] holds head
        // 4 j + tig for the tokens (g, g + 8) of m-tile m
        auto scores = [&](const int cbase, const bool partial, float2 (&lg)[MK][NS]) {
            float acc[MK][NS][2][4];
#pragma unroll
            for (int m = 0; m < MK; ++m)
#pragma unroll
                for (int j = 0; j < NS; ++j)
#pragma unroll
                    for (int u = 0; u < 2; ++u) acc[m][j][u][0] = acc[m][j][u][1] = acc[m][j][u][2] = acc[m][j][u][3] = 0.f;
            {
                // this thread's 32 codes of token cbase + 8 nt + g: word u = channel group u
                uint32_t wl[2 * MK][2], wh[2 * MK][2];
#pragma unroll
                for (int nt = 0; nt < 2 * MK; ++nt) {
                    const uint2 kw = *reinterpret_cast<const uint2*>(pg + kKCodes + (cbase + 8 * nt + g) * 32 + 8 * tig);
                    wl[nt][0] = kw.x;
                    wl[nt][1] = kw.y;
                    wh[nt][0] = kw.x >> 8;
                    wh[nt][1] = kw.y >> 8;
                }
                // k-step 4u + R of every m-tile: A = codes of rows g, g + 8 (n-tiles 2m, 2m + 1)
#define OSCAR_QKT_STEP(R)                                                                                  \
    _Pragma("unroll") for (int m = 0; m < MK; ++m) _Pragma("unroll") for (int u = 0; u < 2; ++u) {        \
        const uint32_t a[4] = {code_pair<R>(wl[2 * m][u]), code_pair<R>(wl[2 * m + 1][u]),                  \
                               code_pair<R>(wh[2 * m][u]), code_pair<R>(wh[2 * m + 1][u])};                 \
        _Pragma("unroll") for (int j = 0; j < NS; ++j)                                                     \
            mma16816(acc[m][j][u], a, qb[j][4 * u + R][0], qb[j][4 * u + R][1]);                          \
    }
                OSCAR_QKT_STEP(0)
                OSCAR_QKT_STEP(1)
                OSCAR_QKT_STEP(2)
                OSCAR_QKT_STEP(3)
#undef OSCAR_QKT_STEP
            }
            // logits: columns (2 tig, 2 tig + 1) of n-tile j are head 4 j + tig's high and low parts
#pragma unroll
            for (int m = 0; m < MK; ++m) {
                const int mt = (cbase >> 4) + m;
                const float4 k0 = sm->tsc[warp][0][mt][g], k1 = sm->tsc[warp][1][mt][g];
#pragma unroll
                for (int j = 0; j < NS; ++j) {
                    const float2 s0 = make_float2(acc[m][j][0][0] + acc[m][j][0][1], acc[m][j][0][2] + acc[m][j][0][3]);
                    const float2 s1 = make_float2(acc[m][j][1][0] + acc[m][j][1][1], acc[m][j][1][2] + acc[m][j][1][3]);
                    float2 x = __ffma2_rn(make_float2(k1.z, k1.w), qs2[j][1], nref[j]);
                    x = __ffma2_rn(make_float2(k0.z, k0.w), qs2[j][0], x);
                    x = __ffma2_rn(make_float2(k1.x, k1.y), s1, x);
                    lg[m][j] = __ffma2_rn(make_float2(k0.x, k0.y), s0, x);
                    if (4 * j + tig >= G) lg[m][j] = make_float2(-INFINITY, -INFINITY);   // no such head
                }
            }
            if (partial) {
                // tokens past the request's end: probability 0 (their scales were staged as 0)
#pragma unroll
                for (int m = 0; m < MK; ++m) {
                    const int t0 = cbase + 16 * m + g;
#pragma unroll
                    for (int j = 0; j < NS; ++j) {
                        if (t0 >= n_live) lg[m][j].x = -INFINITY;
                        if (t0 + 8 >= n_live) lg[m][j].y = -INFINITY;
                    }
                }
            }
        };
        // reference-max update (thread-local test, rare warp-wide raise)
        auto update = [&](float2 (&lg)[MK][NS]) {
            const float tau = sm->tau[warp];
            float cml[NS];
            bool hot = fresh;
#pragma unroll
            for (int j = 0; j < NS; ++j) {
                float cm = -INFINITY;
#pragma unroll
                for (int m = 0; m < MK; ++m) cm = fmaxf(cm, fmaxf(lg[m][j].x, lg[m][j].y));
                cml[j] = cm;
                hot = hot || cm > tau;
            }
            if (__any_sync(0xffffffffu, hot)) {
                float fown[NS], cmx[NS];
#pragma unroll
                for (int j = 0; j < NS; ++j) {
                    // head 4 j + tig's maximum over the warp's row groups (its tokens)
                    float cm = cml[j];
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
                    cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
                    fown[j] = 1.f;
                    cmx[j] = 0.f;
                    if (4 * j + tig < G && (fresh || cm > tau)) {
                        // the reference rises so that the largest logit sits at tau - 7.5
                        const float d = cm - (tau - kTauSlack);
                        fown[j] = fresh ? 0.f : ex2(-d);
                        mref[j] += d;
                        nref[j] = make_float2(-mref[j], -mref[j]);
                        cmx[j] = d;
                        const float2 f2 = make_float2(fown[j], fown[j]);
                        lsum[j] = __fmul2_rn(lsum[j], f2);
                        mv[j][0] = __fmul2_rn(mv[j][0], f2);
                        mv[j][1] = __fmul2_rn(mv[j][1], f2);
                    }
                }
                fresh = false;
#pragma unroll
                for (int m = 0; m < MK; ++m)
#pragma unroll
                    for (int j = 0; j < NS; ++j) lg[m][j] = __fadd2_rn(lg[m][j], make_float2(-cmx[j], -cmx[j]));
                // O^T holds heads 8 mo + 2 tig + e and the page sums head 8 mo + g: head h's factor
                // sits in the lanes with tig = h mod 4, at head tile h / 4
#pragma unroll
                for (int mo = 0; mo < MO; ++mo) {
                    float fo[2], fp;
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int src = (2 * tig + e) & 3;
                        fo[e] = __shfl_sync(0xffffffffu, fown[2 * mo], src);
                        if (2 * mo + 1 < NS) {
                            const float alt = __shfl_sync(0xffffffffu, fown[2 * mo + 1 < NS ? 2 * mo + 1 : 0], src);
                            if (tig >= 2) fo[e] = alt;
                        }
                    }
                    fp = __shfl_sync(0xffffffffu, fown[2 * mo], g & 3);
                    if (2 * mo + 1 < NS) {
                        const float alt = __shfl_sync(0xffffffffu, fown[2 * mo + 1 < NS ? 2 * mo + 1 : 0], g & 3);
                        if (g >= 4) fp = alt;
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        o[c][mo][0] *= fo[0];
                        o[c][mo][1] *= fo[1];
                        o[c][mo][2] *= fo[0];
                        o[c][mo][3] *= fo[1];
                    }
                    psum[mo][0] *= fp;
                    psum[mo][1] *= fp;
                    psum[mo][2] *= fp;
                    psum[mo][3] *= fp;
                }
            }
        };
        // probabilities and P' of one chunk, delivered in the output MMA's B layout
        auto probs = [&](const int cbase, const float2 (&lg)[MK][NS], uint32_t (&pb)[2][KK][MO][2]) {
#pragma unroll
            for (int m = 0; m < MK; ++m) {
                const int mt = (cbase >> 4) + m;
                const float4 v0 = sm->tsc[warp][2][mt][g], v1 = sm->tsc[warp][3][mt][g];
                uint32_t pk[2][NS];      // (P'(t0), P'(t1)) fp16 pairs of head 4 j + tig, value group u
#pragma unroll
                for (int j = 0; j < NS; ++j) {
                    const float2 pr = make_float2(ex2(lg[m][j].x), ex2(lg[m][j].y));
                    lsum[j] = __fadd2_rn(lsum[j], pr);
                    mv[j][0] = __ffma2_rn(pr, make_float2(v0.z, v0.w), mv[j][0]);
                    mv[j][1] = __ffma2_rn(pr, make_float2(v1.z, v1.w), mv[j][1]);
                    const float2 p0 = __fmul2_rn(pr, make_float2(v0.x, v0.y));
                    const float2 p1 = __fmul2_rn(pr, make_float2(v1.x, v1.y));
                    pk[0][j] = pack_h2(p0.x, p0.y);
                    pk[1][j] = pack_h2(p1.x, p1.y);
                }
                // B of k-step m for head tile mo: b0 = P' of tokens 2 tig, 2 tig + 1 (the t0 halves of
                // row groups 2 tig, 2 tig + 1) for head 8 mo + g, b1 = the t1 halves.  Head 8 mo + g
                // is owned by the lanes with tig = g mod 4, at head tile 2 mo + g / 4
                const int srcA = (2 * tig) * 4 + (g & 3), srcB = (2 * tig + 1) * 4 + (g & 3);
#pragma unroll
                for (int u = 0; u < 2; ++u)
#pragma unroll
                    for (int mo = 0; mo < MO; ++mo) {
                        uint32_t xa = __shfl_sync(0xffffffffu, pk[u][2 * mo], srcA);
                        uint32_t xb = __shfl_sync(0xffffffffu, pk[u][2 * mo], srcB);
                        // (heads past the last head tile, g >= 4 there, take copies of real P': their
                        // output columns and page sums are finite and never written out)
                        if (2 * mo + 1 < NS) {
                            const int j1 = 2 * mo + 1 < NS ? 2 * mo + 1 : 0;
                            const uint32_t ya = __shfl_sync(0xffffffffu, pk[u][j1], srcA);
                            const uint32_t yb = __shfl_sync(0xffffffffu, pk[u][j1], srcB);
                            if (g >= 4) xa = ya, xb = yb;
                        }
                        pb[u][m][mo][0] = __byte_perm(xa, xb, 0x5410);
                        pb[u][m][mo][1] = __byte_perm(xa, xb, 0x7632);
                    }
            }
        };
        // O^T += V^T P'^T of one chunk and the page sums of P' (as in decode_mma.cu)
        auto pv = [&](const int cbase, const uint32_t (&pb)[2][KK][MO][2]) {
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
#pragma unroll
            for (int kk = 0; kk < KK; ++kk)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint32_t w0 = vw[q][kk][0], w1 = vw[q][kk][1];
                    const uint32_t s0 = w0 >> 8, s1 = w1 >> 8;
#define OSCAR_PVT_STEP(R)                                                                                \
    {                                                                                                    \
        const uint32_t av[4] = {code_pair<R>(w0), code_pair<R>(s0), code_pair<R>(w1), code_pair<R>(s1)}; \
        _Pragma("unroll") for (int mo = 0; mo < MO; ++mo)                                                \
            mma16816(o[4 * q + R][mo], av, pb[q][kk][mo][0], pb[q][kk][mo][1]);                          \
    }
                    OSCAR_PVT_STEP(0)
                    OSCAR_PVT_STEP(1)
                    OSCAR_PVT_STEP(2)
                    OSCAR_PVT_STEP(3)
#undef OSCAR_PVT_STEP
                }
            // the page's sums of P': A = the output MMAs' B registers in their own order (row g:
            // head g's P' of tokens 0..7, group 0 in k 0..7 and group 1 in k 8..15; row g + 8: tokens
            // 8..15), B = 1 on (k 0..7, columns 0..3) and (k 8..15, columns 4..7)
            const uint32_t sb0 = (g < 4) ? 0x3C003C00u : 0u, sb1 = (g < 4) ? 0u : 0x3C003C00u;
#pragma unroll
            for (int kk = 0; kk < KK; ++kk)
#pragma unroll
                for (int mo = 0; mo < MO; ++mo) {
                    const uint32_t pa[4] = {pb[0][kk][mo][0], pb[0][kk][mo][1], pb[1][kk][mo][0], pb[1][kk][mo][1]};
                    mma16816(psum[mo], pa, sb0, sb1);
                }
        };
        constexpr int NC = kPage / CT;
        if (n_live == kPage) {   // every page but the last of a request: output MMAs of chunk c - 1 after the scores of chunk c
            float2 lg[MK][NS];
            uint32_t pbs[2][2][KK][MO][2];
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
                float2 lg[MK][NS];
                uint32_t pb[2][KK][MO][2];
                scores(cbase, cbase + CT > n_live, lg);
                update(lg);
                probs(cbase, lg, pb);
                pv(cbase, pb);
            }
        }

        // ---- centre the page's output: -1.5 P' per head and value group, in the units of channel
        // tile cm (4^(cm mod 4) 2^-24), then start the next page's sum.  O^T holds heads 2 tig,
        // 2 tig + 1 (+ 8 mo); the sum of head h's group q sits in lane 4 h + 2 q
        float ps_a[MO][2], ps_b[MO][2];
#pragma unroll
        for (int k = 0; k < MO; ++k) {
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
            for (int k = 0; k < MO; ++k) {
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
        for (int k = 0; k < MO; ++k) psum[k][0] = psum[k][1] = psum[k][2] = psum[k][3] = 0.f;

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
            // per-head totals of head 4 j + tig over the warp's row groups
            float m0t[NS], m1t[NS];
#pragma unroll
            for (int j = 0; j < NS; ++j) {
                float l = lsum[j].x + lsum[j].y, m0 = mv[j][0].x + mv[j][0].y, m1 = mv[j][1].x + mv[j][1].y;
#pragma unroll
                for (int o2 = 4; o2 < 32; o2 <<= 1) {
                    l += __shfl_xor_sync(0xffffffffu, l, o2);
                    m0 += __shfl_xor_sync(0xffffffffu, m0, o2);
                    m1 += __shfl_xor_sync(0xffffffffu, m1, o2);
                }
                m0t[j] = m0;
                m1t[j] = m1;
                const int hown = 4 * j + tig;
                if (hown < G && g == 0) {
                    part[(size_t)hown * (2 + kD) + 0] = mref[j];
                    part[(size_t)hown * (2 + kD) + 1] = l;
                }
            }
#pragma unroll
            for (int mo = 0; mo < MO; ++mo)
                // this thread's output entries: heads 8 mo + 2 tig + e, channels 16 cm + g (+ 8); the
                // head's minimum sums sit in the lanes with tig = (2 tig + e) mod 4, at head tile 2 mo + tig / 2
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int hd = 8 * mo + 2 * tig + e;
                    const int src = (2 * tig + e) & 3;
                    float mh0 = __shfl_sync(0xffffffffu, m0t[2 * mo], src);
                    float mh1 = __shfl_sync(0xffffffffu, m1t[2 * mo], src);
                    if (2 * mo + 1 < NS) {
                        const int j1 = 2 * mo + 1 < NS ? 2 * mo + 1 : 0;
                        const float a0 = __shfl_sync(0xffffffffu, m0t[j1], src);
                        const float a1 = __shfl_sync(0xffffffffu, m1t[j1], src);
                        if (tig >= 2) mh0 = a0, mh1 = a1;
                    }
                    if (hd < G) {
                        float* ph = part + (size_t)hd * (2 + kD) + 2;
#pragma unroll
                        for (int cm = 0; cm < 8; ++cm) {
                            // channel tile cm was accumulated at 4^(cm mod 4) * 2^-24 per code
                            const float sc = (float)(1 << (24 - 2 * (cm & 3)));
                            const float mg = cm < 4 ? mh0 : mh1;
                            ph[16 * cm + g] = fmaf(sc, o[cm][mo][e], mg);
                            ph[16 * cm + g + 8] = fmaf(sc, o[cm][mo][2 + e], mg);
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
cudaError_t launch_t_gf(const DecodeParams& p, cudaStream_t s) {
    constexpr int W = warps_t(G);
    const int smem = (int)sizeof(MmaTSmem<W, stages_t(G)>);
    static bool attr_set[kMaxDevices] = {};   // once per instantiation and device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(decode_mma_t<G, FMT64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    decode_mma_t<G, FMT64><<<p.n_units / W, 32 * W, smem, s>>>(p);
    return cudaGetLastError();
}

template <int G>
cudaError_t launch_t_g(const DecodeParams& p, cudaStream_t s) {
    if (p.fmt.gk == 64 && p.fmt.gv == 64) return launch_t_gf<G, true>(p, s);
    return launch_t_gf<G, false>(p, s);
}

}  // namespace

bool decode_mma_t_serves(int g) { return g <= 4 || g == 12; }
int mma_t_units_per_cta(int g) { return warps_t(g); }

cudaError_t launch_decode_mma_t(const DecodeParams& p, cudaStream_t s) {
    switch (p.g) {
        case 1: return launch_t_g<1>(p, s);
        case 2: return launch_t_g<2>(p, s);
        case 3: return launch_t_g<3>(p, s);
        case 4: return launch_t_g<4>(p, s);
        case 12: return launch_t_g<12>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace oscar
