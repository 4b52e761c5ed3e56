// decode_mma.cu -- fused paged GQA decode attention over INT2 pages, warp-level tensor-core MMAs.
//
// The read path of the axbrief.com OSCAR page, section "attention-statistics rotation +
// Triton kernels": keys and values are unpacked and dequantised on chip inside the attention
// pass, with nothing dequantised written back; the key rotation is applied to the query
// (q~ = q . R_K from prep), which equals inverse-rotating every key (R_K orthogonal).
//
// Work split.  The flattened (request, KV head, page) list is cut into equal contiguous runs,
// one per warp PAIR, so every pair streams the same number of bytes whatever the request lengths.
// The two warps of a pair read the same pages and split the 128 channels: warp u owns channel
// group u (channels 64u .. 64u + 63, one quantisation group of 64) for both the scores and the
// output, so each warp holds half of the query fragments and half of the output accumulators.
// Per 32-token chunk (16 for G > 8) the warps swap their partial logits through shared memory
// (one pair barrier), after which both run the same online softmax on the same numbers, so their
// decisions agree exactly.  Warp 0 of the pair keeps a ring of page stages filled by bulk-async
// copies (page-table entries fetched 32 pages ahead); a stage is refilled once both warps have
// moved past its page.  Per page each warp converts its group's fp16 per-token scales and minima
// once into fp32 tables in shared memory.  Per chunk:
//   scores   S_u = Q~_u K_u^T on mma.sync.m16n8k16 (fp16 in, fp32 accumulate): A = the query,
//            rows = head (fp16 high part) and head + 8 (fp16 low part, the rounding residue),
//            so S_hi + S_lo carries ~22 bits of q~; B = 2-bit key codes.  The page stores the
//            codes in fragment order (k_code_byte), so each B register is one AND of a code word
//            (or of the word shifted right by 8) with 0x00030003 << 2r: two fp16 subnormals
//            code * 4^r * 2^-24, exact.  The 4^r of k-step ks (r = ks mod 4) is taken out of the
//            query side (A = q~ * 2^(6 - 2r)), and the query of each (request, KV head) is scaled
//            by a power of two so that its largest high part sits in [2^13, 2^14).  The group's
//            partial logit is 2^18 s_u S_u / qscale + m_u sum_{c in u} q~_c (log2 units);
//   softmax  the two partial logits summed, online, per head, with a lazily raised reference max
//            (output rescaled only when a logit passes the reference by 2^tau, tested per thread
//            first, so the row-group max reduction runs only on that rare path; tau is chosen per
//            segment from the largest value scale so that P' stays inside fp16); all per-token
//            arithmetic runs on packed fp32 pairs (f32x2 FMA / MUL / ADD);
//   output   O_u^T += V_u^T P'_u^T on the same MMA: A = the group's value codes (rows = 16
//            channels), again one AND per register from a 16-byte load in fragment order
//            (v_code_byte), with channel tile r carrying 4^r * 2^-24; B = P' = p * s_V (fp16,
//            columns = 8 heads) straight from the score accumulators' register layout.
//            The dequantised value is m + code * s = (m + 1.5 s) + (code - 1.5) s: the output
//            accumulators take P' (code - 1.5), centred, and the (m + 1.5 s) term runs on the
//            CUDA cores.  The -1.5 P' part is added once per page from the page's sum of P',
//            which one extra MMA per k-step computes exactly as the output MMAs see P' (A = 1).
//            Centring keeps the accumulators near the size of the output itself, so neither the
//            fp16 rounding of P' nor the fp32 accumulation is magnified by a cancellation between
//            two large sums (flat attention over long contexts, peaked attention on one token).
// At the end of each (request, KV head) run the pair writes (reference max, sum, unnormalised
// output) to the split-K partial buffer, one slot per pair.
//
// Waits are bounded: a page-copy wait that gives up sets the error word; the pair agrees on it
// through a barrier reduction and stops, after waiting for its copies still in flight.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx_async.h"

namespace oscar {
namespace {

using namespace ptx;

// Warp pairs per CTA: 8 (16 warps, 128 registers each) when one m-tile holds the G heads
// (G <= 8); 6 (12 warps, 168 registers) for two head tiles.
__host__ __device__ constexpr int pairs_for(int G) { return G <= 8 ? 8 : 6; }
constexpr int kStages = 4;          // page stages per pair
// A raise of the reference max leaves the largest logit this far below tau.  The half step keeps
// the largest probabilities off exact powers of two: with p = 2^k (1 - e) for a nearly flat
// attention, fp16(p * s_V) would round back to the fp16 value 2^k s_V for every token, a
// systematic bias; at 2^(k + 1/2) the rounding errors are spread evenly.
constexpr float kTauSlack = 7.5f;
constexpr float kTauMax = 40.0f;    // tau of a segment before any non-zero value scale is seen
constexpr float kQScaleM = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)

template <int NP>
struct PairSmem {
    uint8_t stage[NP][kStages][kPageHeadBytes];
    uint64_t full[NP][kStages];
    // per warp (channel group u) of a pair, token pairs (2p, 2p + 1) side by side:
    // ktab (2^18 s_K / qscale, same for 2p + 1), (m_K, m_K'); vtab (s_V, s_V'), (m_V + 1.5 s_V, ...)
    float4 ktab[NP][2][32];
    float4 vtab[NP][2][32];
    // partial logits of each group, by chunk parity: [pair][parity][group][head tile x n-tile][lane]
    float2 xch[NP][2][2][4][32];
};

// (request, KV head, page) walk over the flattened page list
struct PageIt {
    int b, h, j, pages;
    __device__ __forceinline__ void init(const DecodeParams& p, int P) {
        int lo = 0, hi = p.batch;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.page_off[mid] <= P) lo = mid;
            else hi = mid;
        }
        b = lo;
        pages = int2_pages(p.len[b]);
        const int rem = P - p.page_off[b];
        h = rem / pages;
        j = rem - h * pages;
    }
    __device__ __forceinline__ bool next(const DecodeParams& p) {   // true when a new segment starts
        if (++j < pages) return false;
        j = 0;
        if (++h == p.hkv) {
            h = 0;
            do {
                ++b;
            } while (b < p.batch - 1 && int2_pages(p.len[b]) == 0);
            if (b >= p.batch) b = p.batch - 1;
            pages = int2_pages(p.len[b]);
        }
        return true;
    }
};

// Wait for a stage's bulk copy: one test, then up to `iters` tests that may each sleep up to 1 ms.
// Gives up (error word set) after that.
__device__ __forceinline__ bool wait_full(uint32_t bar, uint32_t parity, int* err, int iters) {
    if (mbar_try(bar, parity)) return true;
    for (int t = 0; t < iters; ++t)
        if (mbar_try_sleep(bar, parity, 1000000)) return true;
    atomicOr(err, 1);
    return false;
}
constexpr int kDrainIters = 2000;   // copies in flight at a warp's exit: up to about 2 s

// barrier of the 64 threads of one warp pair (named barrier `id`)
__device__ __forceinline__ void pair_sync(int id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }

// the same barrier, returning whether v holds in every thread of the pair
__device__ __forceinline__ bool pair_all(int id, bool v) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, %2, 64, p;\nselp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// codes at bits 2r and 2r + 16 of w as two fp16 subnormals code * 4^r * 2^-24
template <int R>
__device__ __forceinline__ uint32_t code_pair(uint32_t w) { return w & (0x00030003u << (2 * R)); }

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

template <int G>
__global__ void __launch_bounds__(64 * pairs_for(G), 1) decode_mma(const __grid_constant__ DecodeParams p) {
    constexpr int MT = (G + 7) / 8;              // head tiles (rows g and g + 8 of each m-tile)
    constexpr int NT = MT == 1 ? 4 : 2;          // score n-tiles per chunk (8 tokens each)
    constexpr int CT = 8 * NT;                   // tokens per chunk
    constexpr int KK = NT / 2;                   // PV k-steps per chunk
    constexpr int NC = kPage / CT;               // chunks per page
    constexpr int NP = pairs_for(G);
    extern __shared__ __align__(128) uint8_t smem_raw[];
    PairSmem<NP>* sm = reinterpret_cast<PairSmem<NP>*>(smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int pi = warp >> 1, u = warp & 1;      // pair in the CTA, channel group of this warp
    const int bar_id = 1 + pi;
    const int g = lane >> 2, tig = lane & 3;
    const int gp = blockIdx.x * NP + pi;
    const int P0 = (int)(((long long)gp * p.total_pages) / p.n_units);
    const int P1 = (int)(((long long)(gp + 1) * p.total_pages) / p.n_units);
    const int n = P1 - P0;
    if (u == 0 && lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sm->full[pi][s]), 1);
        fence_mbar_init();
    }
    pair_sync(bar_id);   // the stage barriers exist before either warp waits on them
    if (n <= 0) return;

    // ---- page copies (warp 0 of the pair): lane l holds the physical page of page (base + l)
    auto fetch_pt = [&](int base) -> int32_t {
        const int P = P0 + base + lane;
        if (base + lane >= n) return 0;
        PageIt t;
        t.init(p, P);
        return p.page_table[(size_t)t.b * p.max_pps + t.j];
    };
    int pt_base = 0;
    int32_t pt_cur = 0, pt_nxt = 0;
    PageIt is;          // page being issued
    int issued = 0;
    auto issue = [&]() {   // copy page `issued` into its stage
        const int q = issued;
        const int32_t phys = __shfl_sync(0xffffffffu, (q - pt_base) < 32 ? pt_cur : pt_nxt, (q - pt_base) & 31);
        if (lane == 0) {
            const int s = q % kStages;
            const uint32_t bar = smem_u32(&sm->full[pi][s]);
            mbar_expect_tx(bar, p.fmt.bytes);
            bulk_g2s(smem_u32(sm->stage[pi][s]), p.pool + ((size_t)phys * p.hkv + is.h) * p.fmt.bytes, p.fmt.bytes,
                     bar);
        }
        is.next(p);
        ++issued;
    };
    if (u == 0) {
        pt_cur = fetch_pt(0);
        pt_nxt = fetch_pt(32);
        is.init(p, P0);
        for (int k = 0; k < kStages && k < n; ++k) issue();
    }

    // ---- per-segment state (this warp's channel group)
    uint32_t qa[MT][4][4];          // query fragments (hi rows g, lo rows g + 8) per head tile and k-step
    float qs[MT];                   // sum over the group's channels of q~ (logit units)
    float mref[MT];
    float2 lsum[MT], mv[MT];        // per token parity, summed when the partial is written
    bool fresh = true;
    float kscale = 0.f;             // 2^18 / qscale
    float tau = kTauMax, ptau = pow2f((int)kTauMax);
    float o[4][MT][4];              // output^T accumulators: channel tile r (channels 64u + 16r ..), head tile
    float psum[MT][4];              // sum of P' over the current page (rows g, g + 8 alike)
    PageIt it;
    it.init(p, P0);
    bool seg_start = true;
    int chunk_par = 0;

    int consumed = 0;
    for (int i = 0; i < n; ++i) {
        const int s = i % kStages;
        if (seg_start) {
            // power-of-two query scale: the largest |q~| of the group's channels over the G heads,
            // times log2(e) / sqrt(128) * 2^6, lands in [2^13, 2^14), so the fp16 high parts cannot
            // overflow and keep 11 significant bits; exact, and taken out again through kscale and qs
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < MT; ++k) {
                const int hd = g + 8 * k;
                const float* qr = p.qrot + (((size_t)it.b * p.hkv + it.h) * G + (hd < G ? hd : 0)) * kD + 64 * u;
#pragma unroll
                for (int R = 0; R < 4; ++R) {
                    const float2 q0 = *reinterpret_cast<const float2*>(qr + 16 * R + 2 * tig);
                    const float2 q1 = *reinterpret_cast<const float2*>(qr + 16 * R + 2 * tig + 8);
                    if (hd < G) amax = fmaxf(amax, fmaxf(fmaxf(fabsf(q0.x), fabsf(q0.y)), fmaxf(fabsf(q1.x), fabsf(q1.y))));
                }
            }
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
            // floor(log2(amax * log2(e) / sqrt(128) * 64)) from the exponent field, the scale's
            // exponent clamped so that every power of two involved stays a normal fp32 number
            const int ex = (int)((__float_as_uint(amax * (kQScaleM * 64.f)) >> 23) & 0xff) - 127;
            const int e = max(-100, min(100, 13 - ex));
            const float qscale = pow2f(e), qinv = pow2f(-e);
            kscale = pow2f(18 - e);
            // query fragments of this (request, KV head): k-step R of the group holds channels
            // 64u + 16R + 2 tig + (0, 1) (+ 8 for registers 2, 3), scaled by 2^(6 - 2R) against the
            // key codes' 4^R
#pragma unroll
            for (int k = 0; k < MT; ++k) {
                const int hd = g + 8 * k;
                float part = 0.f;
                const float* qr = p.qrot + (((size_t)it.b * p.hkv + it.h) * G + (hd < G ? hd : 0)) * kD + 64 * u;
#pragma unroll
                for (int R = 0; R < 4; ++R) {
                    const float pw = (float)(64 >> (2 * R));      // 2^(6 - 2R), exact
                    const float sc = kQScaleM * pw * qscale, inv = qinv / pw;
                    const float2 q0 = *reinterpret_cast<const float2*>(qr + 16 * R + 2 * tig);
                    const float2 q1 = *reinterpret_cast<const float2*>(qr + 16 * R + 2 * tig + 8);
                    const float qv[2][2] = {{q0.x, q0.y}, {q1.x, q1.y}};
                    float hv[2][2], lv[2][2];
#pragma unroll
                    for (int f = 0; f < 2; ++f)
#pragma unroll
                        for (int e2 = 0; e2 < 2; ++e2) {
                            const float q = hd < G ? qv[f][e2] * sc : 0.f;
                            const float h = __half2float(__float2half_rn(q));
                            const float l = __half2float(__float2half_rn(q - h));
                            hv[f][e2] = h;
                            lv[f][e2] = l;
                            part += (h + l) * inv;
                        }
                    qa[k][R][0] = pack_h2(hv[0][0], hv[0][1]);
                    qa[k][R][1] = pack_h2(lv[0][0], lv[0][1]);
                    qa[k][R][2] = pack_h2(hv[1][0], hv[1][1]);
                    qa[k][R][3] = pack_h2(lv[1][0], lv[1][1]);
                }
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                qs[k] = part;
                mref[k] = 0.f;
                lsum[k] = mv[k] = make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int k = 0; k < MT; ++k) o[r][k][0] = o[r][k][1] = o[r][k][2] = o[r][k][3] = 0.f;
#pragma unroll
            for (int k = 0; k < MT; ++k) psum[k][0] = psum[k][1] = psum[k][2] = psum[k][3] = 0.f;
            seg_start = false;
            fresh = true;
            tau = kTauMax;
            ptau = pow2f((int)kTauMax);
        }
        const bool got = wait_full(smem_u32(&sm->full[pi][s]), (i / kStages) & 1, p.err, p.wait_iters);
        // both warps of the pair take the same decision (a wait may run out in one of them only)
        if (!pair_all(bar_id, __all_sync(0xffffffffu, got))) break;
        consumed = i + 1;
        // both warps are past page i - 1: its stage takes page i - 1 + kStages
        if (u == 0 && i >= 1 && issued < n) {
            if (issued >= pt_base + 32) {
                pt_base += 32;
                pt_cur = pt_nxt;
                pt_nxt = fetch_pt(pt_base + 32);
            }
            issue();
        }
        const uint8_t* pg = sm->stage[pi][s];
        const int n_live = min(kPage, int2_tokens(p.len[it.b]) - it.j * kPage);

        // ---- this group's per-token scales of the page (tokens lane and lane + 32) into fp32 tables.
        // Slots past the request's end are staged as 0 (their bytes may be anything).
        {
            float kv[2][4];
            float vmax = 0.f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = lane + 32 * hh;
                const bool live = t < n_live;
                const uint32_t ksm = p.fmt.gk == 64 ? *reinterpret_cast<const uint32_t*>(pg + kKSm + t * 8 + 4 * u)
                                                    : *reinterpret_cast<const uint32_t*>(pg + kKSm + t * 4);
                uint32_t v0, v1;     // (s, m) of value groups 0 and 1
                if (p.fmt.gv == 64) {
                    const uint2 w = *reinterpret_cast<const uint2*>(pg + p.fmt.v_sm + t * 8);
                    v0 = w.x;
                    v1 = w.y;
                } else {
                    v0 = v1 = *reinterpret_cast<const uint32_t*>(pg + p.fmt.v_sm + t * 4);
                }
                const uint32_t vown = u ? v1 : v0;
                const float sv0 = __half2float(__ushort_as_half(v0 & 0xffff));
                const float sv1 = __half2float(__ushort_as_half(v1 & 0xffff));
                const float sv = __half2float(__ushort_as_half(vown & 0xffff));
                const float mvv = __half2float(__ushort_as_half(vown >> 16));
                vmax = fmaxf(vmax, live ? fmaxf(sv0, sv1) : 0.f);
                kv[hh][0] = live ? kscale * __half2float(__ushort_as_half(ksm & 0xffff)) : 0.f;
                kv[hh][1] = live ? __half2float(__ushort_as_half(ksm >> 16)) : 0.f;
                kv[hh][2] = live ? sv : 0.f;
                kv[hh][3] = live ? fmaf(1.5f, sv, mvv) : 0.f;
            }
            // value scales against the slack: 2^tau * s_V must stay below 2^15 (thread-local test;
            // the warp-wide maximum, the same in both warps, only on the rare path: the first page
            // with non-zero value scales of a segment, or a page whose scales exceed all before)
            if (__any_sync(0xffffffffu, vmax * ptau >= 32768.f)) {
                float w = vmax;
#pragma unroll
                for (int o2 = 1; o2 < 32; o2 <<= 1) w = fmaxf(w, __shfl_xor_sync(0xffffffffu, w, o2));
                // w * 2^tau in [2^14, 2^15): tau = 14 - floor(log2 w) (w > 0 and normal: an fp16 value)
                const int tnew = 14 - ((int)((__float_as_uint(w) >> 23) & 0xff) - 127);
                tau = (float)tnew;
                ptau = pow2f(tnew);
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int t = lane + 32 * hh;
                float* kr = reinterpret_cast<float*>(&sm->ktab[pi][u][t >> 1]);
                float* vr = reinterpret_cast<float*>(&sm->vtab[pi][u][t >> 1]);
                kr[t & 1] = kv[hh][0];
                kr[2 + (t & 1)] = kv[hh][1];
                vr[t & 1] = kv[hh][2];
                vr[2 + (t & 1)] = kv[hh][3];
            }
        }
        __syncwarp();

        // this group's scores and partial logits of one chunk
        auto scores = [&](const int cbase, float2 (&lgo)[MT][NT]) {
            float acc[MT][NT][4];
#pragma unroll
            for (int k = 0; k < MT; ++k)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) acc[k][nt][0] = acc[k][nt][1] = acc[k][nt][2] = acc[k][nt][3] = 0.f;
            {
                // this thread's 16 codes of token cbase + 8 nt + g in the group
                uint32_t wl[NT], wh[NT];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    wl[nt] = *reinterpret_cast<const uint32_t*>(pg + kKCodes + (cbase + 8 * nt + g) * 32 + 8 * tig + 4 * u);
                    wh[nt] = wl[nt] >> 8;
                }
#define OSCAR_QK_STEP(R)                                                                                  \
    _Pragma("unroll") for (int nt = 0; nt < NT; ++nt) {                                                   \
        const uint32_t b0 = code_pair<R>(wl[nt]), b1 = code_pair<R>(wh[nt]);                              \
        _Pragma("unroll") for (int k = 0; k < MT; ++k) mma16816(acc[k][nt], qa[k][R], b0, b1);          \
    }
                OSCAR_QK_STEP(0)
                OSCAR_QK_STEP(1)
                OSCAR_QK_STEP(2)
                OSCAR_QK_STEP(3)
#undef OSCAR_QK_STEP
            }
            // partial logit of the group: kscale s (S_hi + S_lo) + m qs, packed over the token pair
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float4 kt = sm->ktab[pi][u][(cbase >> 1) + 4 * nt + tig];
#pragma unroll
                for (int k = 0; k < MT; ++k) {
                    const float2 hl = __fadd2_rn(make_float2(acc[k][nt][0], acc[k][nt][1]),
                                                 make_float2(acc[k][nt][2], acc[k][nt][3]));
                    lgo[k][nt] = __ffma2_rn(make_float2(kt.x, kt.y), hl,
                                            __fmul2_rn(make_float2(kt.z, kt.w), make_float2(qs[k], qs[k])));
                }
            }
        };
        // publish this group's partial logits of a chunk
        auto publish = [&](const float2 (&lgo)[MT][NT]) {
            float2* xo = &sm->xch[pi][chunk_par][u][0][0];
#pragma unroll
            for (int k = 0; k < MT; ++k)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) xo[(k * NT + nt) * 32 + lane] = lgo[k][nt];
        };
        // full logits (after the pair barrier): own + other - reference; the same in both warps
        auto gather = [&](const int cbase, const bool partial, const float2 (&lgo)[MT][NT], float2 (&lg)[MT][NT]) {
            const float2* xi = &sm->xch[pi][chunk_par][u ^ 1][0][0];
#pragma unroll
            for (int k = 0; k < MT; ++k)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    lg[k][nt] = __fadd2_rn(__fadd2_rn(lgo[k][nt], xi[(k * NT + nt) * 32 + lane]),
                                           make_float2(-mref[k], -mref[k]));
            if (partial) {
                // tokens past the request's end: probability 0
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e2 = 0; e2 < 2; ++e2)
#pragma unroll
                        for (int k = 0; k < MT; ++k)
                            if (cbase + 8 * nt + 2 * tig + e2 >= n_live) (e2 ? lg[k][nt].y : lg[k][nt].x) = -INFINITY;
            }
            chunk_par ^= 1;
        };
        // reference-max update (thread-local test, rare warp-wide raise); the same in both warps
        auto update = [&](float2 (&lg)[MT][NT]) {
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
                        mv[k] = __fmul2_rn(mv[k], f2);
                    }
                }
                fresh = false;
#pragma unroll
                for (int k = 0; k < MT; ++k)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) lg[k][nt] = __fadd2_rn(lg[k][nt], make_float2(-cmx[k], -cmx[k]));
                // O^T and the page's sum of P' hold heads 2 tig, 2 tig + 1 (+ 8 k), whose factors live
                // in the threads of rows g = head
#pragma unroll
                for (int k = 0; k < MT; ++k) {
                    const float f0 = __shfl_sync(0xffffffffu, fown[k], (2 * tig) * 4);
                    const float f1 = __shfl_sync(0xffffffffu, fown[k], (2 * tig + 1) * 4);
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        o[r][k][0] *= f0;
                        o[r][k][1] *= f1;
                        o[r][k][2] *= f0;
                        o[r][k][3] *= f1;
                    }
                    psum[k][0] *= f0;
                    psum[k][1] *= f1;
                    psum[k][2] *= f0;
                    psum[k][3] *= f1;
                }
            }
        };
        // probabilities and this group's P' = p * s_V, rounded once to fp16, packed per token pair
        auto probs = [&](const int cbase, const float2 (&lg)[MT][NT], uint32_t (&pb)[KK][MT][2]) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float4 vt = sm->vtab[pi][u][(cbase >> 1) + 4 * nt + tig];
                const int kk = nt >> 1, half = nt & 1;
#pragma unroll
                for (int k = 0; k < MT; ++k) {
                    const float2 pr = make_float2(ex2(lg[k][nt].x), ex2(lg[k][nt].y));
                    lsum[k] = __fadd2_rn(lsum[k], pr);
                    mv[k] = __ffma2_rn(pr, make_float2(vt.z, vt.w), mv[k]);
                    const float2 pp = __fmul2_rn(pr, make_float2(vt.x, vt.y));
                    pb[kk][k][half] = pack_h2(pp.x, pp.y);
                }
            }
        };
        // O_u^T += V_u^T P'^T of one chunk, and the page's sum of P'
        auto pv = [&](const int cbase, const uint32_t (&pb)[KK][MT][2]) {
            const uint8_t* vsrc = pg + p.fmt.v_codes + 1024 * (cbase >> 5) + 512 * u + 16 * lane;
            uint32_t vw[KK][2];
            if constexpr (KK == 2) {
                const uint4 w4 = *reinterpret_cast<const uint4*>(vsrc);
                vw[0][0] = w4.x;
                vw[0][1] = w4.y;
                vw[1][0] = w4.z;
                vw[1][1] = w4.w;
            } else {
                const uint2 w2 = *reinterpret_cast<const uint2*>(vsrc + 8 * ((cbase >> 4) & 1));
                vw[0][0] = w2.x;
                vw[0][1] = w2.y;
            }
            const uint32_t ones[4] = {0x3C003C00u, 0x3C003C00u, 0x3C003C00u, 0x3C003C00u};   // fp16 1.0
#pragma unroll
            for (int kk = 0; kk < KK; ++kk) {
                const uint32_t w0 = vw[kk][0], w1 = vw[kk][1];
                const uint32_t s0 = w0 >> 8, s1 = w1 >> 8;
#define OSCAR_PV_STEP(R)                                                                                  \
    {                                                                                                     \
        const uint32_t av[4] = {code_pair<R>(w0), code_pair<R>(s0), code_pair<R>(w1), code_pair<R>(s1)};  \
        _Pragma("unroll") for (int k = 0; k < MT; ++k) mma16816(o[R][k], av, pb[kk][k][0], pb[kk][k][1]); \
    }
                OSCAR_PV_STEP(0)
                OSCAR_PV_STEP(1)
                OSCAR_PV_STEP(2)
                OSCAR_PV_STEP(3)
#undef OSCAR_PV_STEP
#pragma unroll
                for (int k = 0; k < MT; ++k) mma16816(psum[k], ones, pb[kk][k][0], pb[kk][k][1]);
            }
        };

        if (n_live == kPage) {
            // every page but the last of a request: the output MMAs of chunk c - 1 run between
            // publishing chunk c's partial logits and the pair barrier
            uint32_t pbs[2][KK][MT][2];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                float2 lgo[MT][NT], lg[MT][NT];
                scores(c * CT, lgo);
                publish(lgo);
                if (c > 0) pv((c - 1) * CT, pbs[(c - 1) & 1]);
                pair_sync(bar_id);
                gather(c * CT, false, lgo, lg);
                update(lg);
                probs(c * CT, lg, pbs[c & 1]);
            }
            pv((NC - 1) * CT, pbs[(NC - 1) & 1]);
        } else {
#pragma unroll
            for (int cbase = 0; cbase < kPage; cbase += CT) {
                if (cbase >= n_live) break;   // the same in both warps
                float2 lgo[MT][NT], lg[MT][NT];
                uint32_t pb[KK][MT][2];
                scores(cbase, lgo);
                publish(lgo);
                pair_sync(bar_id);
                gather(cbase, cbase + CT > n_live, lgo, lg);
                update(lg);
                probs(cbase, lg, pb);
                pv(cbase, pb);
            }
        }
        // centre the page's output: add -1.5 P' (per head, the same for every channel of the
        // group) in the units of channel tile r (4^r 2^-24), then start the next page's sum
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float c = -1.5f * (float)(1 << (2 * r)) * 5.9604644775390625e-08f;   // -1.5 * 4^r * 2^-24
#pragma unroll
            for (int k = 0; k < MT; ++k)
#pragma unroll
                for (int j = 0; j < 4; ++j) o[r][k][j] = fmaf(c, psum[k][j], o[r][k][j]);
        }
#pragma unroll
        for (int k = 0; k < MT; ++k) psum[k][0] = psum[k][1] = psum[k][2] = psum[k][3] = 0.f;

        // this warp is done reading the stage (generic proxy) before a later bulk copy overwrites it
        __syncwarp();
        fence_proxy_async();

        // ---- end of this pair's part of a (request, KV head) run: write the partial result
        const bool last = (i == n - 1);
        const int b_now = it.b, h_now = it.h;
        const bool new_seg = it.next(p);
        if (last || new_seg) {
            float* part = p.part_mma + ((size_t)(b_now * p.hkv + h_now) + gp) * G * (2 + kD);
#pragma unroll
            for (int k = 0; k < MT; ++k) {
                // per-head totals over the four threads of the head's row group
                float l = lsum[k].x + lsum[k].y, m = mv[k].x + mv[k].y;
                l += __shfl_xor_sync(0xffffffffu, l, 1);
                l += __shfl_xor_sync(0xffffffffu, l, 2);
                m += __shfl_xor_sync(0xffffffffu, m, 1);
                m += __shfl_xor_sync(0xffffffffu, m, 2);
                const int hown = g + 8 * k;
                if (u == 0 && hown < G && tig == 0) {
                    part[(size_t)hown * (2 + kD) + 0] = mref[k];
                    part[(size_t)hown * (2 + kD) + 1] = l;
                }
                // this thread's output entries: heads 8 k + 2 tig + e, channels 64 u + 16 r + g (+ 8)
#pragma unroll
                for (int e2 = 0; e2 < 2; ++e2) {
                    const int hd = 8 * k + 2 * tig + e2;
                    const float mh = __shfl_sync(0xffffffffu, m, (2 * tig + e2) * 4);
                    if (hd < G) {
                        float* ph = part + (size_t)hd * (2 + kD) + 2 + 64 * u;
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            // channel tile r was accumulated at 4^r * 2^-24 per code
                            const float sc = (float)(1 << (24 - 2 * r));
                            ph[16 * r + g] = fmaf(sc, o[r][k][e2], mh);
                            ph[16 * r + g + 8] = fmaf(sc, o[r][k][2 + e2], mh);
                        }
                    }
                }
            }
            seg_start = true;
        }
    }
    // copies still in flight must land before the warp may exit (only after a timeout)
    if (u == 0 && lane == 0)
        for (int q = consumed; q < issued; ++q)
            wait_full(smem_u32(&sm->full[pi][q % kStages]), (q / kStages) & 1, p.err, kDrainIters);
}

template <int G>
cudaError_t launch_mma_g(const DecodeParams& p, cudaStream_t s) {
    constexpr int NP = pairs_for(G);
    const int smem = (int)sizeof(PairSmem<NP>);
    static bool attr_set[kMaxDevices] = {};   // once per instantiation and device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(decode_mma<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    decode_mma<G><<<p.n_units / NP, 64 * NP, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int mma_units_per_cta(int g) { return pairs_for(g); }

cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t s) {
    if (p.total_pages == 0) return cudaSuccess;
    count_launches(1);
    switch (p.g) {
        case 1: return launch_mma_g<1>(p, s);
        case 2: return launch_mma_g<2>(p, s);
        case 3: return launch_mma_g<3>(p, s);
        case 4: return launch_mma_g<4>(p, s);
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
