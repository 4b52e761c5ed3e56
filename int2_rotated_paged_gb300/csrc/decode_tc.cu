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
// whatever the request lengths.  Sixteen warps in four warpgroups:
//   WG0, WG1  token groups (thread = token = TMEM lane), alternating tiles: unpack the tile's
//             2-bit key codes to fp16 (1 + code/4) into their own TMEM A buffer, then run
//             the online softmax of that tile on their own score and output accumulators:
//             logit = sum_g 4 s_g S_g + (m_g - 4 s_g) sum_{c in g} q~_c, a reference max that
//             is raised only when a logit passes it by 2^8 (then O is rescaled once),
//             P' = p * s_V per head and group stored as the B operand of the PV product;
//   WG2       value group (thread = channel = TMEM lane): unpacks the tile's channel-major
//             value codes into a 3-deep ring of TMEM A buffers;
//   WG3       warp 12 producer (bulk-async copies of each tile's two 5120-byte page blocks into
//             a 10-stage shared-memory ring, page-table entries fetched a batch ahead),
//             warp 13 issues S = A_K x Q^T (M 128 tokens, N 16, q split into fp16 hi and lo
//             halves that two MMAs add into one accumulator per 64-channel group), warp 14
//             issues O += A_V x P'^T (M 128 channels, K tokens, N = 2G padded), all
//             tcgen05.mma kind::f16 with A read from TMEM, fp32 accumulators in TMEM.
// Each token group writes its own (reference max, sum, unnormalised output) per segment (a
// run of tiles of one request and KV head); combine (decode.cu) merges them with the BF16
// sink / window part.
//
// Every mbarrier wait is bounded (about two seconds of clock cycles); on timeout the kernel
// records an error word, stops waiting, drains its own copies and MMAs, frees its tensor
// memory and returns.  Warp-uniform roles never leave their loops early, so named barriers
// and .sync.aligned instructions always see every thread.
#include <cuda_fp16.h>

#include "internal.h"
#include "tc_ptx.h"

namespace oscar {
namespace {

using namespace ptx;

constexpr int kThreads = 512;
constexpr int kStages = 10;
constexpr int kNV = 3;                                   // value A-buffer ring depth
constexpr int kStageBytes = 2 * kPageHeadBytes;
constexpr float kTau = 8.0f;
constexpr float kQScale = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)

// TMEM columns
constexpr uint32_t kColAK = 0;      // 2 x 64  (token group w)
constexpr uint32_t kColAV = 128;    // 3 x 64
constexpr uint32_t kColS = 320;     // 2 x 32  (group 0: 16 columns, group 1: 16 columns)
constexpr uint32_t kColO = 384;     // 2 x 32
constexpr uint32_t kTmemCols = 512;

// shared memory
constexpr uint32_t kQLbo = 128, kQSbo = 2048;    // Q: K-major, 16 rows x 128 k per half
constexpr uint32_t kQHalf = 4096;                 // hi half, then lo half
constexpr uint32_t kQBuf = 2 * kQHalf;            // one buffer per segment parity
// P': MN-major (N contiguous).  The K-group stride is padded from 128 to 144 bytes so that the
// eight tokens of a quarter-warp (even or odd K rows of two groups) hit distinct banks.
constexpr uint32_t kPLbo = 144, kPSbo = 16 * 144;
constexpr uint32_t kPBuf = 4 * kPSbo;             // up to 32 rows
constexpr int kOffQ = kStages * kStageBytes;
constexpr int kOffP = kOffQ + 2 * kQBuf;
constexpr int kOffMisc = kOffP + 2 * kPBuf;

struct Misc {
    uint64_t full[kStages], empty[kStages];
    uint64_t akf[2], sf[2], pf[2], pe[2], of[2], oe[2];
    uint64_t avf[kNV], ave[kNV];
    uint64_t qf[2], qe[2];
    uint64_t drain_q, drain_p;
    uint32_t tmem;
    int abort_flag;
    float qsum[2][kMaxG][2];
    float redm[2][4][kMaxG];
    float red5[2][4][kMaxG * 5];
    float qred[2][4][kMaxG];
};
constexpr int kSmemBytes = kOffMisc + (int)sizeof(Misc);

// Walks the CTA's tiles in order: request b, KV head h, tile j of (b, h), and the local
// indices of the first and last tile of the current segment.
struct TileIt {
    int i, b, h, j, tiles, seg, sfirst, slast, n;

    __device__ __forceinline__ void init(const DecodeParams& p, int T0, int n_) {
        n = n_;
        i = 0;
        int lo = 0, hi = p.batch;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.tile_off[mid] <= T0) lo = mid;
            else hi = mid;
        }
        b = lo;
        tiles = int2_tiles(p.len[b]);
        const int rem = T0 - p.tile_off[b];
        h = rem / tiles;
        j = rem - h * tiles;
        seg = 0;
        sfirst = 0;
        slast = min(n - 1, tiles - 1 - j);
    }
    __device__ __forceinline__ void next(const DecodeParams& p) {
        ++i;
        if (++j == tiles) {
            j = 0;
            if (++h == p.hkv) {
                h = 0;
                do {
                    ++b;
                } while (b < p.batch - 1 && int2_tiles(p.len[b]) == 0);
                tiles = int2_tiles(p.len[b < p.batch ? b : p.batch - 1]);
            }
            ++seg;
            sfirst = i;
            slast = min(n - 1, i + tiles - 1);
        }
    }
};

// Bounded wait: the thread sleeps in try_wait (up to 1 ms per attempt, woken when the phase
// completes), at most kWaitTries attempts.  False (abort flag set, error word written) on
// timeout; once the CTA has aborted, waits return false at once unless `drain` is set (tail
// waits for copies and MMAs in flight, which must land before the CTA may exit).
constexpr uint32_t kSleepNs = 1000000;
constexpr int kWaitTries = 2000;
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Misc* m, int* err, bool drain = false) {
    if (mbar_try_sleep(bar, parity, kSleepNs)) return true;
    for (int t = 1; t < kWaitTries; ++t) {
        if (!drain && *(volatile int*)&m->abort_flag) return false;
        if (mbar_try_sleep(bar, parity, kSleepNs)) return true;
    }
    *(volatile int*)&m->abort_flag = 1;
    atomicOr(err, 1);
    return false;
}

// fp16x2 (1 + code_a / 4, 1 + code_b / 4) of the two codes at bits 2R and 2R + 16 of w.
template <int R>
__device__ __forceinline__ uint32_t half_pair(uint32_t w) {
    uint32_t x;
    if constexpr (R < 4) x = w << (8 - 2 * R);
    else if constexpr (R == 4) x = w;
    else x = w >> (2 * R - 8);
    return (x & 0x03000300u) | 0x3C003C00u;
}

template <int I, int N>
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t (&v)[N]) {
    v[8 * I + 0] = half_pair<0>(w);
    v[8 * I + 1] = half_pair<1>(w);
    v[8 * I + 2] = half_pair<2>(w);
    v[8 * I + 3] = half_pair<3>(w);
    v[8 * I + 4] = half_pair<4>(w);
    v[8 * I + 5] = half_pair<5>(w);
    v[8 * I + 6] = half_pair<6>(w);
    v[8 * I + 7] = half_pair<7>(w);
}

// 64 codes (16 bytes) -> 32 fp16x2 words
__device__ __forceinline__ void unpack64(uint4 a, uint32_t (&v)[32]) {
    unpack_word<0>(a.x, v);
    unpack_word<1>(a.y, v);
    unpack_word<2>(a.z, v);
    unpack_word<3>(a.w, v);
}

// 128 codes -> two 32-column TMEM stores (keeps only 32 words live at a time)
__device__ __forceinline__ void unpack_store128(uint4 a, uint4 b, uint32_t taddr) {
    uint32_t v[32];
    unpack64(a, v);
    tmem_st32(taddr, v);
    unpack64(b, v);
    tmem_st32(taddr + 32, v);
}

// K position of element x of the unpacked order: codes (r, r + 8) of each 16-code word share
// TMEM column r, i.e. K positions 2r and 2r + 1 of that 16-element block.
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

template <int NPV>
__device__ __forceinline__ void ld_o(uint32_t taddr, uint32_t (&v)[NPV]) {
    if constexpr (NPV == 16) tmem_ld16(taddr, v);
    else tmem_ld32(taddr, v);
}
template <int NPV>
__device__ __forceinline__ void st_o(uint32_t taddr, const uint32_t (&v)[NPV]) {
    if constexpr (NPV == 16) tmem_st16(taddr, v);
    else tmem_st32(taddr, v);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1) decode_tc(const __grid_constant__ DecodeParams p) {
    constexpr int NPV = ((2 * G + 15) / 16) * 16;                  // N of the PV product
    constexpr uint32_t kIdescQK = idesc_f16(128, 16);
    constexpr uint32_t kIdescPV = idesc_f16(128, NPV) | (1u << 16);   // B (P') is MN-major
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc* m = reinterpret_cast<Misc*>(smem + kOffMisc);
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int T0 = (int)(((long long)blockIdx.x * p.total_tiles) / p.n_cta);
    const int T1 = (int)(((long long)(blockIdx.x + 1) * p.total_tiles) / p.n_cta);
    const int n = T1 - T0;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&m->full[s]), 1);
            mbar_init(smem_u32(&m->empty[s]), 256);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(smem_u32(&m->akf[x]), 128);
            mbar_init(smem_u32(&m->sf[x]), 1);
            mbar_init(smem_u32(&m->pf[x]), 128);
            mbar_init(smem_u32(&m->pe[x]), 1);
            mbar_init(smem_u32(&m->of[x]), 1);
            mbar_init(smem_u32(&m->oe[x]), 128);
            mbar_init(smem_u32(&m->qf[x]), 128);
            mbar_init(smem_u32(&m->qe[x]), 1);
        }
        for (int x = 0; x < kNV; ++x) {
            mbar_init(smem_u32(&m->avf[x]), 128);
            mbar_init(smem_u32(&m->ave[x]), 1);
        }
        mbar_init(smem_u32(&m->drain_q), 1);
        mbar_init(smem_u32(&m->drain_p), 1);
        m->abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = tid; i < (2 * kQBuf + 2 * kPBuf) / 16; i += kThreads)
        reinterpret_cast<uint4*>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
    if (warp == 13) tmem_alloc(smem_u32(&m->tmem), kTmemCols);
    fence_proxy_async();
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tm = m->tmem;

    // Register split: the token groups take 184 per thread, the value group keeps 88 and the
    // producer / MMA group 56 (184 + 184 + 88 + 56 = 4 x 128, the launch's reservation).  The
    // only increase is the token groups' one below, so it is always granted from what the other
    // groups release; nothing gives registers back before exit.
    if (warp >= 12) {
        regs_dec<56>();
        if (warp == 12) {
            // ============================================================ producer
            constexpr int kBatch = 16;
            TileIt it;      // tile described by lane (2k, 2k + 1) of the batch being fetched
            it.init(p, T0, n);
            TileIt is = it; // tile being issued
            auto fetch = [&](TileIt& f, int count) -> int32_t {
                // lanes 2k and 2k + 1 fetch the two page ids of the k-th tile of the batch
                int32_t v = 0;
                for (int k = 0; k < count; ++k) {
                    if (lane >> 1 == k) {
                        const int pg = 2 * f.j + (lane & 1);
                        if (pg < int2_pages(p.len[f.b])) v = p.page_table[(size_t)f.b * p.max_pps + pg];
                    }
                    f.next(p);
                }
                return v;
            };
            int32_t cur = fetch(it, min(kBatch, n));
            bool ok = true;
            int issued = 0;
            for (int base = 0; base < n && ok; base += kBatch) {
                const int cnt = min(kBatch, n - base);
                const int nxt_cnt = min(kBatch, n - base - cnt);
                const int32_t nxt = nxt_cnt > 0 ? fetch(it, nxt_cnt) : 0;
                for (int k = 0; k < cnt; ++k) {
                    const int i = base + k;
                    const int32_t ph0 = __shfl_sync(0xffffffffu, cur, 2 * k);
                    const int32_t ph1 = __shfl_sync(0xffffffffu, cur, 2 * k + 1);
                    if (lane == 0) {
                        const int s = i % kStages;
                        const int use = i / kStages;
                        if (use > 0 && !wait_bar(smem_u32(&m->empty[s]), (use - 1) & 1, m, p.err)) ok = false;
                        if (ok) {
                            const bool two = 2 * is.j + 1 < int2_pages(p.len[is.b]);
                            const uint32_t bar = smem_u32(&m->full[s]);
                            const uint32_t dst = smem_u32(smem + s * kStageBytes);
                            mbar_expect_tx(bar, two ? 2 * kPageHeadBytes : kPageHeadBytes);
                            bulk_g2s(dst, p.pool + ((size_t)ph0 * p.hkv + is.h) * kPageHeadBytes, kPageHeadBytes, bar);
                            if (two)
                                bulk_g2s(dst + kPageHeadBytes, p.pool + ((size_t)ph1 * p.hkv + is.h) * kPageHeadBytes,
                                         kPageHeadBytes, bar);
                            issued = i + 1;
                        }
                    }
                    is.next(p);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                }
                cur = nxt;
            }
            if (lane == 0)
                for (int i = max(0, issued - kStages); i < issued; ++i)
                    wait_bar(smem_u32(&m->full[i % kStages]), (i / kStages) & 1, m, p.err, true);
        } else if (warp == 13) {
            // ============================================================ QK issuer
            if (lane == 0) {
                TileIt it;
                it.init(p, T0, n);
                const uint32_t qbase = smem_u32(smem + kOffQ);
                for (int i = 0; i < n; ++i) {
                    const int w = i & 1;
                    if (i == it.sfirst && !wait_bar(smem_u32(&m->qf[it.seg & 1]), (it.seg >> 1) & 1, m, p.err)) break;
                    if (!wait_bar(smem_u32(&m->akf[w]), (i >> 1) & 1, m, p.err)) break;
                    tc_after();
                    const uint32_t qa = qbase + (it.seg & 1) * kQBuf;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint32_t d = tm + kColS + 32 * w + 16 * (ks >> 2);
                        const uint32_t a = tm + kColAK + 64 * w + 8 * ks;
                        umma_ts(d, a, sdesc(qa + ks * 2 * kQLbo, kQLbo, kQSbo), kIdescQK, (ks & 3) != 0);
                        umma_ts(d, a, sdesc(qa + kQHalf + ks * 2 * kQLbo, kQLbo, kQSbo), kIdescQK, 1);
                    }
                    umma_commit(smem_u32(&m->sf[w]));
                    if (i == it.slast) umma_commit(smem_u32(&m->qe[it.seg & 1]));
                    it.next(p);
                }
                umma_commit(smem_u32(&m->drain_q));
                wait_bar(smem_u32(&m->drain_q), 0, m, p.err, true);
            }
            __syncwarp();
        } else if (warp == 14) {
            // ============================================================ PV issuer
            if (lane == 0) {
                TileIt it;
                it.init(p, T0, n);
                int started[2] = {0, 0};
                const uint32_t pbase = smem_u32(smem + kOffP);
                for (int i = 0; i < n; ++i) {
                    const int w = i & 1, x = i % kNV;
                    const bool first = i - it.sfirst <= 1;
                    const bool last = it.slast - i <= 1;
                    if (!wait_bar(smem_u32(&m->avf[x]), (i / kNV) & 1, m, p.err)) break;
                    if (!wait_bar(smem_u32(&m->pf[w]), (i >> 1) & 1, m, p.err)) break;
                    if (first && started[w] > 0 &&
                        !wait_bar(smem_u32(&m->oe[w]), (started[w] - 1) & 1, m, p.err))
                        break;
                    if (first) ++started[w];
                    tc_after();
                    const uint32_t pa = pbase + w * kPBuf;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_ts(tm + kColO + 32 * w, tm + kColAV + 64 * x + 8 * ks,
                                sdesc(pa + ks * 2 * kPLbo, kPLbo, kPSbo), kIdescPV, !(first && ks == 0));
                    umma_commit(smem_u32(&m->ave[x]));
                    umma_commit(smem_u32(&m->pe[w]));
                    if (last) umma_commit(smem_u32(&m->of[w]));
                    it.next(p);
                }
                umma_commit(smem_u32(&m->drain_p));
                wait_bar(smem_u32(&m->drain_p), 0, m, p.err, true);
            }
            __syncwarp();
        }
    } else if (warp >= 8) {
        // ================================================================ value group
        regs_dec<88>();
        const int r = tid - 256;
        const uint32_t lanebase = (uint32_t)(32 * (warp - 8)) << 16;
        for (int i = 0; i < n; ++i) {
            const int s = i % kStages, x = i % kNV, use = i / kNV;
            wait_bar(smem_u32(&m->full[s]), (i / kStages) & 1, m, p.err);
            const uint8_t* st = smem + s * kStageBytes;
            const uint4 x0 = *reinterpret_cast<const uint4*>(st + kVCodes + r * 16);
            const uint4 x1 = *reinterpret_cast<const uint4*>(st + kPageHeadBytes + kVCodes + r * 16);
            mbar_arrive(smem_u32(&m->empty[s]));
            if (use > 0) wait_bar(smem_u32(&m->ave[x]), (use - 1) & 1, m, p.err);
            tc_after();
            unpack_store128(x0, x1, tm + lanebase + kColAV + 64 * x);
            tmem_wait_st();
            tc_before();
            mbar_arrive(smem_u32(&m->avf[x]));
        }
    } else {
        // ================================================================ token groups
        regs_inc<184>();
        const int w = warp >> 2;             // token group
        const int wk = warp & 3;             // warp within the group
        const int r = tid - 128 * w;         // token of the tile = TMEM lane
        const uint32_t lanebase = (uint32_t)(32 * wk) << 16;
        const int bar_vote = 1 + 2 * w, bar_sync_id = 2 + 2 * w;
        const int kq = kpos(r);
        const uint32_t pdst = smem_u32(smem + kOffP + w * kPBuf) + (kq >> 3) * kPLbo + (kq & 7) * 16;
        constexpr bool kQsRegs = G <= 12;       // G = 16 reads the per-group q sums from shared memory
        float mref[G], l[G], sp[G][2], mv[G][2], qs[kQsRegs ? G : 1][2];
        int flushes = 0;
        TileIt it;
        it.init(p, T0, n);
        if (w == 1 && n > 1) it.next(p);
        for (int i = w; i < n; i += 2) {
            const int s = i % kStages;
            const int k = i >> 1;                           // this group's tile count so far
            const bool first = i - it.sfirst <= 1;
            const bool last = it.slast - i <= 1;
            const int qpar = it.seg & 1;
            if (i == it.sfirst) {
                // ---- this group opens the segment: Q operand (hi / lo fp16) and per-group sums
                if (it.seg >= 2) wait_bar(smem_u32(&m->qe[qpar]), ((it.seg - 2) >> 1) & 1, m, p.err);
                const float* qr = p.qrot + ((size_t)it.b * p.hkv * G + (size_t)it.h * G) * kD;
                uint8_t* Q = smem + kOffQ + qpar * kQBuf;
                const int kc = kq >> 3, kin = kq & 7;
                float part[G];
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float q = qr[hh * kD + r] * kQScale;
                    const __half hi = __float2half_rn(q);
                    const __half lo = __float2half_rn(q - __half2float(hi));
                    const int off = (hh >> 3) * kQSbo + kc * kQLbo + (hh & 7) * 16 + kin * 2;
                    *reinterpret_cast<__half*>(Q + off) = hi;
                    *reinterpret_cast<__half*>(Q + kQHalf + off) = lo;
                    part[hh] = warp_sum(__half2float(hi) + __half2float(lo));
                }
                if (lane == 0)
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) m->qred[w][wk][hh] = part[hh];
                bar_sync(bar_sync_id, 128);
                if (r < G) {
                    m->qsum[qpar][r][0] = m->qred[w][0][r] + m->qred[w][1][r];
                    m->qsum[qpar][r][1] = m->qred[w][2][r] + m->qred[w][3][r];
                }
                fence_proxy_async();
                mbar_arrive(smem_u32(&m->qf[qpar]));
            }
            if (first) {
                if (i != it.sfirst) wait_bar(smem_u32(&m->qf[qpar]), (it.seg >> 1) & 1, m, p.err);
                else bar_sync(bar_sync_id, 128);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    if constexpr (kQsRegs) {
                        qs[hh][0] = m->qsum[qpar][hh][0];
                        qs[hh][1] = m->qsum[qpar][hh][1];
                    }
                    mref[hh] = -INFINITY;
                    l[hh] = 0.f;
                    sp[hh][0] = sp[hh][1] = mv[hh][0] = mv[hh][1] = 0.f;
                }
            }
            // ---- keys of token r -> TMEM A operand
            wait_bar(smem_u32(&m->full[s]), (i / kStages) & 1, m, p.err);
            const uint8_t* st = smem + s * kStageBytes + (r >> 6) * kPageHeadBytes;
            {
                // 32 bytes per token: lanes with (r >> 2) odd read the upper half first, so each
                // quarter-warp's 16-byte loads cover all 32 banks
                const uint8_t* src = st + kKCodes + (r & 63) * 32;
                const int sw = (r >> 2) & 1;
                const uint4 y0 = *reinterpret_cast<const uint4*>(src + 16 * sw);
                const uint4 y1 = *reinterpret_cast<const uint4*>(src + 16 * (sw ^ 1));
                const uint4 x0 = sw ? y1 : y0, x1 = sw ? y0 : y1;
                tc_after();
                unpack_store128(x0, x1, tm + lanebase + kColAK + 64 * w);
                tmem_wait_st();
                tc_before();
                mbar_arrive(smem_u32(&m->akf[w]));
            }
            const uint2 ksm = *reinterpret_cast<const uint2*>(st + kKSm + (r & 63) * 8);
            const uint2 vsm = *reinterpret_cast<const uint2*>(st + kVSm + (r & 63) * 8);
            mbar_arrive(smem_u32(&m->empty[s]));
            const bool live = it.j * kTileTok + r < int2_tokens(p.len[it.b]);
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
            // ---- scores
            wait_bar(smem_u32(&m->sf[w]), k & 1, m, p.err);
            tc_after();
            uint32_t sv[32];
            tmem_ld32(tm + lanebase + kColS + 32 * w, sv);
            tmem_wait_ld();
            float lg[G];
            bool ex = false;
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float q0, q1;
                if constexpr (kQsRegs) {
                    q0 = qs[hh][0];
                    q1 = qs[hh][1];
                } else {
                    q0 = m->qsum[qpar][hh][0];
                    q1 = m->qsum[qpar][hh][1];
                }
                float x = fmaf(a0, __uint_as_float(sv[hh]),
                               fmaf(a1, __uint_as_float(sv[16 + hh]), fmaf(c0, q0, c1 * q1)));
                x = live ? x : -INFINITY;
                lg[hh] = x;
                ex |= x > mref[hh] + kTau;
            }
            // ---- raise the reference max when a logit passes it by more than 2^8 (rare)
            if (bar_or(bar_vote, 128, ex)) {
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float tmx = warp_max(lg[hh]);
                    if (lane == 0) m->redm[w][wk][hh] = tmx;
                }
                bar_sync(bar_sync_id, 128);
                float f[G];
                bool changed = false;
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float tmx = fmaxf(fmaxf(m->redm[w][0][hh], m->redm[w][1][hh]),
                                            fmaxf(m->redm[w][2][hh], m->redm[w][3][hh]));
                    const float old = mref[hh];
                    const float nw = (tmx > old + kTau) ? tmx : old;
                    f[hh] = (old == -INFINITY) ? 0.f : exp2f(old - nw);
                    changed |= nw != old;
                    mref[hh] = nw;
                }
                bar_sync(bar_sync_id, 128);
                if (changed && !first) {
                    // O holds this group's earlier tiles: rescale once its last PV is done
                    wait_bar(smem_u32(&m->pe[w]), (k - 1) & 1, m, p.err);
                    tc_after();
                    uint32_t o[NPV];
                    ld_o<NPV>(tm + lanebase + kColO + 32 * w, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 2 * G; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f[c >> 1]);
                    st_o<NPV>(tm + lanebase + kColO + 32 * w, o);
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
            // ---- probabilities, P' = p * s_V (fp16, N contiguous) for the PV product
            uint32_t pp[NPV / 2];
#pragma unroll
            for (int c = 0; c < NPV / 2; ++c) pp[c] = 0u;
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float pr = live ? exp2f(lg[hh] - mref[hh]) : 0.f;
                l[hh] += pr;
                const __half2 h2 = __floats2half2_rn(pr * vs0, pr * vs1);
                sp[hh][0] += __low2float(h2);
                sp[hh][1] += __high2float(h2);
                mv[hh][0] = fmaf(pr, vm0, mv[hh][0]);
                mv[hh][1] = fmaf(pr, vm1, mv[hh][1]);
                pp[hh] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            if (k > 0) wait_bar(smem_u32(&m->pe[w]), (k - 1) & 1, m, p.err);
#pragma unroll
            for (int c = 0; c < NPV / 8; ++c)
                st_shared_v4(pdst + c * kPSbo, pp[4 * c], pp[4 * c + 1], pp[4 * c + 2], pp[4 * c + 3]);
            fence_proxy_async();
            tc_before();
            mbar_arrive(smem_u32(&m->pf[w]));

            // ---- this group's last tile of the segment: write its partial result
            if (last) {
                wait_bar(smem_u32(&m->of[w]), flushes & 1, m, p.err);
                ++flushes;
                tc_after();
                uint32_t o[NPV];
                ld_o<NPV>(tm + lanebase + kColO + 32 * w, o);
                tmem_wait_ld();
                tc_before();
                mbar_arrive(smem_u32(&m->oe[w]));
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float v0 = warp_sum(l[hh]);
                    const float v1 = warp_sum(sp[hh][0]);
                    const float v2 = warp_sum(sp[hh][1]);
                    const float v3 = warp_sum(mv[hh][0]);
                    const float v4 = warp_sum(mv[hh][1]);
                    if (lane == 0) {
                        m->red5[w][wk][5 * hh + 0] = v0;
                        m->red5[w][wk][5 * hh + 1] = v1;
                        m->red5[w][wk][5 * hh + 2] = v2;
                        m->red5[w][wk][5 * hh + 3] = v3;
                        m->red5[w][wk][5 * hh + 4] = v4;
                    }
                }
                bar_sync(bar_sync_id, 128);
                const int gc = r >> 6;
                float* part = p.part_tc + (((size_t)(it.b * p.hkv + it.h) + blockIdx.x) * 2 + w) * G * (2 + kD);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float tot[5];
#pragma unroll
                    for (int q = 0; q < 5; ++q)
                        tot[q] = m->red5[w][0][5 * hh + q] + m->red5[w][1][5 * hh + q] + m->red5[w][2][5 * hh + q] +
                                 m->red5[w][3][5 * hh + q];
                    const float spg = gc ? tot[2] : tot[1];
                    const float mvg = gc ? tot[4] : tot[3];
                    part[hh * (2 + kD) + 2 + r] = fmaf(4.f, __uint_as_float(o[2 * hh + gc]) - spg, mvg);
                    if (r == 0) {
                        part[hh * (2 + kD) + 0] = mref[hh];
                        part[hh * (2 + kD) + 1] = tot[0];
                    }
                }
                bar_sync(bar_sync_id, 128);
            }
            it.next(p);
            if (i + 1 < n) it.next(p);
        }
    }

    // ---- tear-down: every role is past its last wait; free the tensor memory
    tc_before();
    __syncthreads();
    tc_after();
    if (warp == 13) tmem_dealloc(tm, kTmemCols);
}

template <int G>
cudaError_t launch_g(const DecodeParams& p, cudaStream_t s) {
    // The warpgroups' setmaxnreg targets (184 + 184 + 88 + 56) add up to 4 x 128: the launch
    // must reserve exactly 128 registers per thread or the increase could never be granted.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, decode_tc<G>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != 128) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(decode_tc<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
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
