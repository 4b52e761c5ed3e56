// decode_tc.cu -- fused paged GQA decode attention over INT2 pages on the sm_103a tensor cores.
//
// The read path of the axbrief.com OSCAR page, section "attention-statistics rotation +
// Triton kernels": INT2 keys and values are unpacked and dequantised on chip, attention runs
// in one pass, and nothing dequantised is written back to global memory.  The key rotation
// is applied to the query (q~ = q . R_K, computed by rotate_q); scores use q~ against the
// rotated keys, which equals inverse-rotating every key because R_K is orthogonal.
//
// One persistent CTA per SM walks a contiguous range of 128-token tiles (two INT2 pages) of
// the flattened (request, KV head, tile) list, so every SM streams the same number of bytes
// whatever the request lengths.  Roles (10 warps):
//   warp 8      producer: bulk-async copies of each tile's two 5120-byte page blocks into a
//               10-stage shared-memory ring (page-table entries fetched one batch ahead);
//   warps 0-3   dequant: thread = TMEM lane.  Keys: thread = token, its 128 2-bit codes become
//               64 fp16x2 words (1 + code/4) stored to TMEM; values (channel-major pages):
//               thread = channel, its 128 tokens' codes likewise;
//   warp 9      MMA: S = A_K x Q^T (M = 128 tokens, N = 2G padded: q split in fp16 hi + lo,
//               one accumulator per 64-channel group) and O += A_V x P'^T (M = 128 channels,
//               K = tokens, N = 2G: p * s_V per head and group), tcgen05.mma kind::f16 with A
//               read from TMEM and B from shared memory, fp32 accumulators in TMEM;
//   warps 4-7   softmax: thread = token.  logit = sum_g 4 s_g S_g + (m_g - 4 s_g) sum_g(q~),
//               online softmax with a lazily raised reference (rescale O only when a logit
//               exceeds the reference by 2^8), P' stores for the PV MMA, and the per-segment
//               flush out = sum_t p m_V + 4 (O - sum_t P') of each (request, KV head) run.
// A segment's result (reference max, sum, unnormalised output) goes to the split-K partial
// buffer; combine (decode.cu) merges segments and the BF16 sink / window part.
//
// Every wait on an mbarrier is bounded (about two seconds of clock cycles); on timeout the
// kernel records an error word, stops issuing work, drains its own copies and MMAs, frees
// its tensor memory and returns.
#include <cuda_fp16.h>

#include "internal.h"
#include "tc_ptx.h"

namespace oscar {
namespace {

using namespace ptx;

constexpr int kWarps = 10;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 10;
constexpr int kStageBytes = 2 * kPageHeadBytes;
constexpr float kTau = 8.0f;
constexpr float kQScale = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
constexpr long long kWaitCycles = 4000000000ll;

constexpr uint32_t kColAK = 0, kColAV = 128, kColS = 256, kColO = 384, kTmemCols = 512;
constexpr uint32_t kQLbo = 128, kQSbo = 2048;          // Q operand core-matrix strides (K, N)
constexpr uint32_t kPLbo = 144, kPSbo = 16 * 144;      // P' operand: padded K stride

constexpr int kOffQ = kStages * kStageBytes;
constexpr int kQBytes = 4 * kQSbo;
constexpr int kOffP = kOffQ + kQBytes;
constexpr int kPBytes = 4 * kPSbo;
constexpr int kOffMisc = kOffP + 2 * kPBytes;

struct Misc {
    uint64_t full[kStages], empty[kStages];
    uint64_t akf[2], ake[2], avf[2], ave[2], sf[2], se[2], pf[2], pe[2];
    uint64_t qf, qe, of, oe, drain;
    uint32_t tmem;
    int abort_flag;
    float redm[4][kMaxG];
    float red5[4][kMaxG * 5];
    float qred[4][kMaxG];
};
constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc);

struct Tile {
    int b, h, j, tiles;
};

__device__ __forceinline__ Tile tile_at(const DecodeParams& p, int T) {
    int lo = 0, hi = p.batch;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.tile_off[mid] <= T) lo = mid;
        else hi = mid;
    }
    Tile t;
    t.b = lo;
    t.tiles = int2_tiles(p.len[lo]);
    const int rem = T - p.tile_off[lo];
    t.h = rem / t.tiles;
    t.j = rem - t.h * t.tiles;
    return t;
}

// Bounded wait: false (and the CTA abort flag set, the error word written) on timeout.  Once the
// CTA has aborted, waits return false at once unless `drain` is set (the tail waits for copies and
// MMAs in flight, which must land before the CTA may exit; those stay bounded by the timeout).
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, Misc* m, int* err, bool drain = false) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try(bar, parity)) return true;
        if (!drain && *(volatile int*)&m->abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            *(volatile int*)&m->abort_flag = 1;
            atomicOr(err, 1);
            return false;
        }
    }
}

// fp16x2 (1 + code_a / 4, 1 + code_b / 4) of the two codes at bits 2r and 2r + 16 of w.
template <int R>
__device__ __forceinline__ uint32_t half_pair(uint32_t w) {
    uint32_t x;
    if constexpr (R < 4) x = w << (8 - 2 * R);
    else if constexpr (R == 4) x = w;
    else x = w >> (2 * R - 8);
    return (x & 0x03000300u) | 0x3C003C00u;
}

template <int I>
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t (&v)[64]) {
    v[8 * I + 0] = half_pair<0>(w);
    v[8 * I + 1] = half_pair<1>(w);
    v[8 * I + 2] = half_pair<2>(w);
    v[8 * I + 3] = half_pair<3>(w);
    v[8 * I + 4] = half_pair<4>(w);
    v[8 * I + 5] = half_pair<5>(w);
    v[8 * I + 6] = half_pair<6>(w);
    v[8 * I + 7] = half_pair<7>(w);
}

__device__ __forceinline__ void unpack128(uint4 a, uint4 b, uint32_t (&v)[64]) {
    unpack_word<0>(a.x, v);
    unpack_word<1>(a.y, v);
    unpack_word<2>(a.z, v);
    unpack_word<3>(a.w, v);
    unpack_word<4>(b.x, v);
    unpack_word<5>(b.y, v);
    unpack_word<6>(b.z, v);
    unpack_word<7>(b.w, v);
}

// Position in the MMA's K order of element u of a 16-element block: the unpack pairs
// elements (r, r + 8) of each 16-code word into TMEM column r, i.e. K positions 2r, 2r + 1.
__device__ __forceinline__ int kpos(int x) { return (x & ~15) + 2 * (x & 7) + ((x >> 3) & 1); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

template <int NP>
__device__ __forceinline__ void ld_cols(uint32_t taddr, uint32_t (&v)[NP]) {
    if constexpr (NP == 16) tmem_ld16(taddr, v);
    else if constexpr (NP == 32) tmem_ld32(taddr, v);
    else tmem_ld64(taddr, v);
}
template <int NP>
__device__ __forceinline__ void st_cols(uint32_t taddr, const uint32_t (&v)[NP]) {
    if constexpr (NP == 16) tmem_st16(taddr, v);
    else if constexpr (NP == 32) tmem_st32(taddr, v);
    else tmem_st64(taddr, v);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1) decode_tc(const __grid_constant__ DecodeParams p) {
    constexpr int NP = ((2 * G + 15) / 16) * 16;   // MMA N (both products)
    constexpr uint32_t kIdesc = idesc_f16(128, NP);
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc* m = reinterpret_cast<Misc*>(smem + kOffMisc);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int T0 = (int)(((long long)blockIdx.x * p.total_tiles) / p.n_cta);
    const int T1 = (int)(((long long)(blockIdx.x + 1) * p.total_tiles) / p.n_cta);
    const int n = T1 - T0;

    // ---- set-up: barriers, TMEM, zeroed operand buffers
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&m->full[s]), 1);
            mbar_init(smem_u32(&m->empty[s]), 256);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_u32(&m->akf[x]), 128);
            mbar_init(smem_u32(&m->ake[x]), 1);
            mbar_init(smem_u32(&m->avf[x]), 128);
            mbar_init(smem_u32(&m->ave[x]), 1);
            mbar_init(smem_u32(&m->sf[x]), 1);
            mbar_init(smem_u32(&m->se[x]), 128);
            mbar_init(smem_u32(&m->pf[x]), 128);
            mbar_init(smem_u32(&m->pe[x]), 1);
        }
        mbar_init(smem_u32(&m->qf), 128);
        mbar_init(smem_u32(&m->qe), 1);
        mbar_init(smem_u32(&m->of), 1);
        mbar_init(smem_u32(&m->oe), 128);
        mbar_init(smem_u32(&m->drain), 1);
        m->abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = tid; i < (kQBytes + 2 * kPBytes) / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
    if (warp == 9) tmem_alloc(smem_u32(&m->tmem), kTmemCols);
    fence_proxy_async();
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tm = m->tmem;

    if (warp == 8) {
        // ================================================================ producer
        constexpr int kBatch = 16;
        auto fetch = [&](int bi) -> int32_t {
            const int i = bi * kBatch + (lane >> 1);
            if (i >= n) return 0;
            const Tile t = tile_at(p, T0 + i);
            const int pg = 2 * t.j + (lane & 1);
            if (pg >= int2_pages(p.len[t.b])) return 0;
            return p.page_table[(size_t)t.b * p.max_pps + pg];
        };
        const int nb = (n + kBatch - 1) / kBatch;
        int32_t cur = nb > 0 ? fetch(0) : 0;
        bool ok = true;
        int issued = 0;
        for (int bi = 0; bi < nb && ok; ++bi) {
            const int32_t nxt = (bi + 1 < nb) ? fetch(bi + 1) : 0;
            for (int k = 0; k < kBatch; ++k) {
                const int i = bi * kBatch + k;
                if (i >= n) break;
                const int32_t ph0 = __shfl_sync(0xffffffffu, cur, 2 * k);
                const int32_t ph1 = __shfl_sync(0xffffffffu, cur, 2 * k + 1);
                if (lane == 0) {
                    const int s = i % kStages;
                    const int use = i / kStages;
                    if (use > 0 && !wait_bar(smem_u32(&m->empty[s]), (use - 1) & 1, m, p.err)) ok = false;
                    if (ok) {
                        const Tile t = tile_at(p, T0 + i);
                        const bool two = 2 * t.j + 1 < int2_pages(p.len[t.b]);
                        const uint32_t bar = smem_u32(&m->full[s]);
                        const uint32_t dst = smem_u32(smem + s * kStageBytes);
                        mbar_expect_tx(bar, two ? 2 * kPageHeadBytes : kPageHeadBytes);
                        bulk_g2s(dst, p.pool + ((size_t)ph0 * p.hkv + t.h) * kPageHeadBytes, kPageHeadBytes, bar);
                        if (two)
                            bulk_g2s(dst + kPageHeadBytes, p.pool + ((size_t)ph1 * p.hkv + t.h) * kPageHeadBytes,
                                     kPageHeadBytes, bar);
                        issued = i + 1;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            cur = nxt;
        }
        // every issued copy must have landed before the CTA may exit
        if (lane == 0) {
            for (int i = max(0, issued - kStages); i < issued; ++i)
                wait_bar(smem_u32(&m->full[i % kStages]), (i / kStages) & 1, m, p.err, true);
        }
    } else if (warp == 9) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t qaddr = smem_u32(smem + kOffQ);
            int seg = 0;        // segment of the QK tile
            int pseg = 0;       // segment of the PV tile
            bool ok = true;
            for (int i = 0; i <= n && ok; ++i) {
                if (i < n) {
                    const Tile t = tile_at(p, T0 + i);
                    if (i > 0 && t.j == 0) ++seg;
                    const int a = i & 1, use = i >> 1;
                    if (t.j == 0 || i == 0) ok = ok && wait_bar(smem_u32(&m->qf), seg & 1, m, p.err);
                    ok = ok && wait_bar(smem_u32(&m->akf[a]), use & 1, m, p.err);
                    if (use > 0) ok = ok && wait_bar(smem_u32(&m->se[a]), (use - 1) & 1, m, p.err);
                    if (!ok) break;
                    tc_after();
                    const uint32_t d0 = tm + kColS + 64 * a;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_ts(d0 + (ks < 4 ? 0 : NP), tm + kColAK + 64 * a + 8 * ks,
                                sdesc(qaddr + ks * 2 * kQLbo, kQLbo, kQSbo), kIdesc, (ks & 3) != 0);
                    umma_commit(smem_u32(&m->sf[a]));
                    umma_commit(smem_u32(&m->ake[a]));
                    if (t.j == t.tiles - 1 || i == n - 1) umma_commit(smem_u32(&m->qe));
                }
                if (i >= 1) {
                    const int i2 = i - 1;
                    const Tile t = tile_at(p, T0 + i2);
                    const bool first = (t.j == 0) || i2 == 0;
                    if (i2 > 0 && t.j == 0) ++pseg;
                    const int a = i2 & 1, use = i2 >> 1;
                    ok = ok && wait_bar(smem_u32(&m->avf[a]), use & 1, m, p.err);
                    ok = ok && wait_bar(smem_u32(&m->pf[a]), use & 1, m, p.err);
                    if (first && pseg > 0) ok = ok && wait_bar(smem_u32(&m->oe), (pseg - 1) & 1, m, p.err);
                    if (!ok) break;
                    tc_after();
                    const uint32_t paddr = smem_u32(smem + kOffP + a * kPBytes);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_ts(tm + kColO, tm + kColAV + 64 * a + 8 * ks,
                                sdesc(paddr + ks * 2 * kPLbo, kPLbo, kPSbo), kIdesc, !(first && ks == 0));
                    umma_commit(smem_u32(&m->ave[a]));
                    umma_commit(smem_u32(&m->pe[a]));
                    if (t.j == t.tiles - 1 || i2 == n - 1) umma_commit(smem_u32(&m->of));
                }
            }
            // all issued MMAs must finish before the tensor memory is released
            umma_commit(smem_u32(&m->drain));
            wait_bar(smem_u32(&m->drain), 0, m, p.err, true);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ================================================================ dequant (thread = TMEM lane)
        const int r = tid;
        const uint32_t lanebase = (uint32_t)(32 * warp) << 16;
        for (int i = 0; i < n; ++i) {
            const int s = i % kStages;
            wait_bar(smem_u32(&m->full[s]), (i / kStages) & 1, m, p.err);
            const uint8_t* st = smem + s * kStageBytes;
            const int a = i & 1, use = i >> 1;
            uint32_t v[64];
            {   // keys: token r, 32 bytes of codes
                const uint4* src = reinterpret_cast<const uint4*>(st + (r >> 6) * kPageHeadBytes + kKCodes + (r & 63) * 32);
                const uint4 x0 = src[0], x1 = src[1];
                unpack128(x0, x1, v);
            }
            if (use > 0) wait_bar(smem_u32(&m->ake[a]), (use - 1) & 1, m, p.err);
            tc_after();
            tmem_st64(tm + lanebase + kColAK + 64 * a, v);
            tmem_wait_st();
            tc_before();
            mbar_arrive(smem_u32(&m->akf[a]));
            {   // values: channel r, 16 bytes (64 tokens) from each page
                const uint4 x0 = *reinterpret_cast<const uint4*>(st + kVCodes + r * 16);
                const uint4 x1 = *reinterpret_cast<const uint4*>(st + kPageHeadBytes + kVCodes + r * 16);
                unpack128(x0, x1, v);
            }
            if (use > 0) wait_bar(smem_u32(&m->ave[a]), (use - 1) & 1, m, p.err);
            tc_after();
            tmem_st64(tm + lanebase + kColAV + 64 * a, v);
            tmem_wait_st();
            tc_before();
            mbar_arrive(smem_u32(&m->avf[a]));
            mbar_arrive(smem_u32(&m->empty[s]));
        }
    } else {
        // ================================================================ softmax (thread = token / channel lane)
        const int w4 = warp - 4;
        const int r = tid - 128;
        const uint32_t lanebase = (uint32_t)(32 * w4) << 16;
        const int kq = kpos(r);
        float mref[G], l[G], sp[G][2], mv[G][2], qs[G][2];
        auto reset = [&]() {
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                mref[hh] = -INFINITY;
                l[hh] = 0.f;
                sp[hh][0] = sp[hh][1] = mv[hh][0] = mv[hh][1] = 0.f;
            }
        };
        // Q operand of the segment that starts at local tile i (channel r of every head)
        auto write_q = [&](const Tile& t) {
            const float* qr = p.qrot + ((size_t)t.b * p.hkv * G + (size_t)t.h * G) * kD;
            uint8_t* Q = smem + kOffQ;
            const int kc = kq >> 3, kin = kq & 7;
            float part[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float q = qr[hh * kD + r] * kQScale;
                const __half hi = __float2half_rn(q);
                const __half lo = __float2half_rn(q - __half2float(hi));
                const int n0 = 2 * hh, n1 = 2 * hh + 1;
                *reinterpret_cast<__half*>(Q + (n0 >> 3) * kQSbo + kc * kQLbo + (n0 & 7) * 16 + kin * 2) = hi;
                *reinterpret_cast<__half*>(Q + (n1 >> 3) * kQSbo + kc * kQLbo + (n1 & 7) * 16 + kin * 2) = lo;
                part[hh] = warp_sum(__half2float(hi) + __half2float(lo));
            }
            if (lane == 0)
#pragma unroll
                for (int hh = 0; hh < G; ++hh) m->qred[w4][hh] = part[hh];
            bar_sync(2, 128);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                qs[hh][0] = m->qred[0][hh] + m->qred[1][hh];
                qs[hh][1] = m->qred[2][hh] + m->qred[3][hh];
            }
            bar_sync(2, 128);
            fence_proxy_async();
            mbar_arrive(smem_u32(&m->qf));
        };
        reset();
        if (n > 0) write_q(tile_at(p, T0));
        int seg = 0;
        // Warp-uniform roles never leave the loop early: after an abort every wait returns at
        // once and all 128 threads still meet at the same named barriers.
        for (int i = 0; i < n; ++i) {
            const Tile t = tile_at(p, T0 + i);
            const bool first = (t.j == 0) || i == 0;
            const int s = i % kStages;
            const int a = i & 1, use = i >> 1;
            // ---- scores of this tile (TMEM -> registers)
            wait_bar(smem_u32(&m->sf[a]), use & 1, m, p.err);
            tc_after();
            uint32_t sv[2 * NP];
            if constexpr (NP == 16) {
                tmem_ld32(tm + lanebase + kColS + 64 * a, sv);
            } else {
                tmem_ld64(tm + lanebase + kColS + 64 * a, sv);
            }
            tmem_wait_ld();
            tc_before();
            mbar_arrive(smem_u32(&m->se[a]));
            wait_bar(smem_u32(&m->full[s]), (i / kStages) & 1, m, p.err);
            const uint8_t* st = smem + s * kStageBytes + (r >> 6) * kPageHeadBytes;
            const uint2 ksm = *reinterpret_cast<const uint2*>(st + kKSm + (r & 63) * 8);
            const uint2 vsm = *reinterpret_cast<const uint2*>(st + kVSm + (r & 63) * 8);
            mbar_arrive(smem_u32(&m->empty[s]));
            const bool live = t.j * kTileTok + r < int2_tokens(p.len[t.b]);
            const float ks0 = __half2float(__ushort_as_half(ksm.x & 0xffff));
            const float km0 = __half2float(__ushort_as_half(ksm.x >> 16));
            const float ks1 = __half2float(__ushort_as_half(ksm.y & 0xffff));
            const float km1 = __half2float(__ushort_as_half(ksm.y >> 16));
            const float vs0 = live ? __half2float(__ushort_as_half(vsm.x & 0xffff)) : 0.f;
            const float vm0 = live ? __half2float(__ushort_as_half(vsm.x >> 16)) : 0.f;
            const float vs1 = live ? __half2float(__ushort_as_half(vsm.y & 0xffff)) : 0.f;
            const float vm1 = live ? __half2float(__ushort_as_half(vsm.y >> 16)) : 0.f;
            const float a0 = 4.f * ks0, a1 = 4.f * ks1;
            const float c0 = km0 - a0, c1 = km1 - a1;
            float lg[G];
            bool ex = false;
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float t0 = __uint_as_float(sv[2 * hh]) + __uint_as_float(sv[2 * hh + 1]);
                const float t1 = __uint_as_float(sv[NP + 2 * hh]) + __uint_as_float(sv[NP + 2 * hh + 1]);
                float x = fmaf(a0, t0, fmaf(a1, t1, fmaf(c0, qs[hh][0], c1 * qs[hh][1])));
                x = live ? x : -INFINITY;
                lg[hh] = x;
                ex |= x > mref[hh] + kTau;
            }
            // ---- raise the reference max when a logit passes it by more than 2^8 (rare)
            if (bar_or(1, 128, ex)) {
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float tmx = warp_max(lg[hh]);
                    if (lane == 0) m->redm[w4][hh] = tmx;
                }
                bar_sync(2, 128);
                float f[G];
                bool changed = false;
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float tmx = fmaxf(fmaxf(m->redm[0][hh], m->redm[1][hh]), fmaxf(m->redm[2][hh], m->redm[3][hh]));
                    const float old = mref[hh];
                    const float nw = (tmx > old + kTau) ? tmx : old;
                    f[hh] = (old == -INFINITY) ? 0.f : exp2f(old - nw);
                    changed |= nw != old;
                    mref[hh] = nw;
                }
                bar_sync(2, 128);
                if (changed && !first) {
                    // O holds earlier tiles of this segment: rescale it once PV(i - 1) is done
                    wait_bar(smem_u32(&m->pe[(i - 1) & 1]), ((i - 1) >> 1) & 1, m, p.err);
                    tc_after();
                    uint32_t o[NP];
                    ld_cols<NP>(tm + lanebase + kColO, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 2 * G; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f[c >> 1]);
                    st_cols<NP>(tm + lanebase + kColO, o);
                    tmem_wait_st();
                    tc_before();
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        l[hh] *= f[hh];
                        sp[hh][0] *= f[hh];
                        sp[hh][1] *= f[hh];
                        mv[hh][0] *= f[hh];
                        mv[hh][1] *= f[hh];
                    }
                }
            }
            // ---- probabilities, P' = p * s_V (fp16) for the PV MMA
            if (use > 0) wait_bar(smem_u32(&m->pe[a]), (use - 1) & 1, m, p.err);
            uint8_t* P = smem + kOffP + a * kPBytes + (kq >> 3) * kPLbo + (kq & 7) * 2;
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float pr = live ? exp2f(lg[hh] - mref[hh]) : 0.f;
                l[hh] += pr;
                const __half2 h2 = __floats2half2_rn(pr * vs0, pr * vs1);
                sp[hh][0] += __low2float(h2);
                sp[hh][1] += __high2float(h2);
                mv[hh][0] = fmaf(pr, vm0, mv[hh][0]);
                mv[hh][1] = fmaf(pr, vm1, mv[hh][1]);
                const int n0 = 2 * hh, n1 = 2 * hh + 1;
                *reinterpret_cast<__half*>(P + (n0 >> 3) * kPSbo + (n0 & 7) * 16) = __low2half(h2);
                *reinterpret_cast<__half*>(P + (n1 >> 3) * kPSbo + (n1 & 7) * 16) = __high2half(h2);
            }
            fence_proxy_async();
            mbar_arrive(smem_u32(&m->pf[a]));

            // ---- end of a (request, KV head) segment: write its partial result
            if (t.j == t.tiles - 1 || i == n - 1) {
                if (i + 1 < n) {
                    wait_bar(smem_u32(&m->qe), seg & 1, m, p.err);
                    write_q(tile_at(p, T0 + i + 1));
                }
                wait_bar(smem_u32(&m->of), seg & 1, m, p.err);
                tc_after();
                uint32_t o[NP];
                ld_cols<NP>(tm + lanebase + kColO, o);
                tmem_wait_ld();
                tc_before();
                mbar_arrive(smem_u32(&m->oe));
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float v0 = warp_sum(l[hh]);
                    const float v1 = warp_sum(sp[hh][0]);
                    const float v2 = warp_sum(sp[hh][1]);
                    const float v3 = warp_sum(mv[hh][0]);
                    const float v4 = warp_sum(mv[hh][1]);
                    if (lane == 0) {
                        m->red5[w4][5 * hh + 0] = v0;
                        m->red5[w4][5 * hh + 1] = v1;
                        m->red5[w4][5 * hh + 2] = v2;
                        m->red5[w4][5 * hh + 3] = v3;
                        m->red5[w4][5 * hh + 4] = v4;
                    }
                }
                bar_sync(2, 128);
                const int gc = r >> 6;
                float* part = p.part_tc + ((size_t)(t.b * p.hkv + t.h) + blockIdx.x) * G * (2 + kD);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float tot[5];
#pragma unroll
                    for (int q = 0; q < 5; ++q)
                        tot[q] = m->red5[0][5 * hh + q] + m->red5[1][5 * hh + q] + m->red5[2][5 * hh + q] +
                                 m->red5[3][5 * hh + q];
                    const float spg = gc ? tot[2] : tot[1];
                    const float mvg = gc ? tot[4] : tot[3];
                    const float out = fmaf(4.f, __uint_as_float(o[2 * hh + gc]) - spg, mvg);
                    part[hh * (2 + kD) + 2 + r] = out;
                    if (r == 0) {
                        part[hh * (2 + kD) + 0] = mref[hh];
                        part[hh * (2 + kD) + 1] = tot[0];
                    }
                }
                bar_sync(2, 128);
                reset();
                ++seg;
            }
        }
    }

    // ---- tear-down: every role is past its last wait; free the tensor memory
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == 9) tmem_dealloc(tm, kTmemCols);
}

template <int G>
cudaError_t launch_g(const DecodeParams& p, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    decode_tc<G><<<p.n_cta, kThreads, kSmemBytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t s) {
    if (p.total_tiles == 0) return cudaSuccess;
    count_launches(1);
    switch (p.g) {
        case 1: return launch_g<1>(p, s);
        case 2: return launch_g<2>(p, s);
        case 3: return launch_g<3>(p, s);
        case 4: return launch_g<4>(p, s);
        case 5: return launch_g<5>(p, s);
        case 6: return launch_g<6>(p, s);
        case 7: return launch_g<7>(p, s);
        case 8: return launch_g<8>(p, s);
        case 12: return launch_g<12>(p, s);
        case 16: return launch_g<16>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace oscar
