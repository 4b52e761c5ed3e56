// prep.cu -- first kernel of a warp-MMA decode call, one CTA per (KV head, request).  Its
// prep_step form (oscar_decode_step) first appends the request's new token for the KV head: the
// token leaving the window is read, the new one written into the slot it leaves, and the leaving
// key, rotated in the same R_K loop as the queries, is quantised into its INT2 slot.  Then:
//   1. q~ = q . R_K for the G query heads of the KV head (fp32), the queries of the INT2 pages
//      (axbrief.com OSCAR page, section "attention-statistics rotation + Triton kernels": scores
//      against rotated keys; rotating q once equals inverse-rotating every key, R_K orthogonal);
//   2. attention of the plain queries over the request's BF16 sink + window tokens (same page,
//      section "OSCAR release": BF16 sink and recent window), written as one split-K partial
//      (reference max, sum, unnormalised output) that combine merges with the INT2 partials.
// Scores of the BF16 part run on mma.sync m16n8k16 with bf16 operands: A = the query (rows: the
// bf16 high part of 8 heads, then their bf16 low parts, ~16 bits in all), B = key rows (a fragment
// register is two adjacent channels of one token).  Each warp takes every kPrepWarps-th 8-slot tile
// and stages its K and V rows in two shared-memory buffers by asynchronous copies, the first two
// tiles requested before the query rotation so that their loads overlap it.  The online softmax
// runs per warp over the tiles; P.V runs on the CUDA cores with the probabilities shared through
// shared memory (lane = 4 output channels).
// All softmax arithmetic is in base 2 (logits pre-scaled by log2(e) / sqrt(128)).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx_async.h"
#include "token_quant.h"

namespace oscar {
namespace {

// warps per CTA: 8 when the per-warp output partials of G <= 8 heads fit in static shared memory
__host__ __device__ constexpr int prep_warps(int G) { return G <= 8 ? 8 : 4; }
// BF16 sink / window tiles of 8 slots, staged per warp in two buffers by asynchronous copies: K and V
// rows padded to 272 bytes (the 8 rows of an MMA fragment load or of an ldmatrix fall on all 32 banks)
constexpr int kKRow = 272;
constexpr int kTileBytes = 16 * kKRow;
__host__ __device__ constexpr int prep_dyn_smem(int G) { return prep_warps(G) * 2 * kTileBytes; }
constexpr float kQScaleP = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)

__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

__device__ __forceinline__ float load_query(const DecodeParams& p, size_t idx) {
    return p.q_dtype == 0 ? reinterpret_cast<const float*>(p.q)[idx]
                          : bf16_to_f(reinterpret_cast<const uint16_t*>(p.q)[idx]);
}

__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// m16n8k8 with bf16 operands: A = rows g, g + 8 at k 2 tig, 2 tig + 1; B = k 2 tig, 2 tig + 1 of column g
__device__ __forceinline__ void mma_bf16_k8(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

// four 8 x 8 b16 matrices from shared memory, transposed: lanes 8 i .. 8 i + 7 give the row addresses
// of matrix i; matrix i's element (row 2 tig + e, column g) lands in half e of register i of lane (g, tig)
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// slot s of the BF16 region holds a token of a request of length len
__device__ __forceinline__ bool slot_live(int s, int n_sink, int n_win) {
    return s < n_sink || (s >= kSink && s < kSink + n_win);
}

// STEP: the CTA first appends request b's new token for KV head h (the fused decode step, one new
// token per request): the token leaving the window is read, the new one written into its BF16 slot,
// and the leaving key is rotated in the same loop as the queries and quantised into its INT2 slot.
template <int G, bool STEP>
__device__ __forceinline__ void prep_body(const DecodeParams& p, const AppendParams* ap) {
    constexpr int MT = (G + 7) / 8;                  // head tiles (rows g and g + 8 of each)
    constexpr int kPrepWarps = prep_warps(G);
    constexpr int NT = 32 * kPrepWarps;
    __shared__ float qs[G][kD];                      // plain queries
    __shared__ float mw[kPrepWarps][G], lw[kPrepWarps][G];
    __shared__ float ow[kPrepWarps][G][kD];
    const int h = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
    const int warp = c >> 5, lane = c & 31, g = lane >> 2, tig = lane & 3;
    if (b == 0 && h == 0 && c == 0 && p.err) {
        *p.err = 0;
        if (p.wait_probe) {
            // timeout-path check: a bounded wait on a barrier that nothing arrives at runs out and
            // sets the error word, exactly as a page copy that never lands would
            __shared__ uint64_t probe;
            const uint32_t bar = ptx::smem_u32(&probe);
            ptx::mbar_init(bar, 1);
            ptx::fence_mbar_init();
            bool done = ptx::mbar_try(bar, 0);
            for (int t = 0; t < p.wait_iters && !done; ++t) done = ptx::mbar_try_sleep(bar, 0, 1000000);
            if (!done) atomicOr(p.err, 1);
        }
    }
    const size_t qbase = ((size_t)b * p.hkv + h) * G * kD;

    __shared__ float xk[STEP ? kD : 1];              // key leaving the window (fp32)
    __shared__ float red[2 * kPrepWarps];
    __shared__ uint8_t tpart[2][4][16];              // packing scratch of the leaving token
    const bool evict = STEP && ap->req[b].e1 > ap->req[b].e0;   // the same for the whole CTA
    float yv = 0.f;
    if constexpr (STEP) {
        const AppendReq& r = ap->req[b];
        if (evict && c < kD) {
            xk[c] = tq::bf16_bits_to_f32(tq::token_src(*ap, b, h, 0, r.e0)[c]);
            yv = tq::bf16_bits_to_f32(tq::token_src(*ap, b, h, 1, r.e0)[c]);
        }
        __syncthreads();   // read before the new token takes the slot it leaves
        for (int i = c; i < 2 * kD; i += NT) {
            const int kv = i / kD, ch = i % kD;
            const uint16_t* src = (kv == 0 ? ap->k : ap->v) + ((size_t)r.tok_off * p.hkv + h) * kD;
            ap->bf16[((((size_t)b * p.hkv + h) * 2 + kv) * kSlots + bf16_slot(r.len0)) * kD + ch] = src[ch];
        }
        if (h == 0 && c == 0) ap->seq_lens[b] = r.len0 + r.n_new;
    }
    // query row r of the slot: query token r / g_real (of the slot's nq) and head h * g_real + r % g_real
    // of the caller's layout [rows][hkv * g_real][128]; rows of missing query tokens are zero
    for (int i = c; i < G * kD; i += NT) {
        const int r = i / kD, j = r / p.g_real;
        qs[r][i % kD] = j < p.nq[b] ? load_query(p, (((size_t)p.q0[b] + j) * p.hkv * p.g_real + (size_t)h * p.g_real +
                                                     r % p.g_real) * kD + i % kD)
                                    : 0.f;
    }
    __syncthreads();

    // ---- this warp's BF16 tiles (8 slots each: tiles warp, warp + kPrepWarps, ...): the first two
    // are requested now, so that their loads overlap the query rotation; tile i + 2 is requested
    // once tile i has been used (one commit group per tile, empty ones included)
    extern __shared__ __align__(16) uint8_t prep_dyn[];
    uint8_t* wbuf = prep_dyn + (size_t)warp * 2 * kTileBytes;
    const uint16_t* kb = p.bf16 + (((size_t)p.row[b] * p.hkv + h) * 2 + 0) * kSlots * kD;
    const uint16_t* vb = p.bf16 + (((size_t)p.row[b] * p.hkv + h) * 2 + 1) * kSlots * kD;
    const int len = p.len[b];
    const int n_sink = min(len, kSink), n_win = min(kWindow, max(0, len - kSink));
    constexpr int kTiles = (kSlots / 8 + kPrepWarps - 1) / kPrepWarps;
    auto tile_used = [&](int nt) {
        return nt < kSlots / 8 && (slot_live(8 * nt, n_sink, n_win) || slot_live(8 * nt + 7, n_sink, n_win));
    };
    auto request_tile = [&](int i) {
        const int nt = warp + kPrepWarps * i;
        if (i < kTiles && tile_used(nt)) {
            const uint32_t dst = ptx::smem_u32(wbuf + (i & 1) * kTileBytes);
            // 8 rows x 256 bytes of K, then of V: 256 pieces of 16 bytes, 8 per lane
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int piece = lane + 32 * j, kv = piece >> 7, row = (piece >> 4) & 7, ch = piece & 15;
                const uint16_t* src = (kv ? vb : kb) + (size_t)(8 * nt + row) * kD + 8 * ch;
                const uint32_t d = dst + (kv ? 8 * kKRow : 0) + kKRow * row + 16 * ch;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
            }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    request_tile(0);
    request_tile(1);

    // ---- q~[i][col] = sum_j q[i][j] R_h[j][col]: column col of R_h, 32 rows in flight.  With 8
    // warps the two halves of the CTA split the rows (each R_K entry is loaded once per CTA) and
    // add their partial sums; with 4 warps one thread takes a whole column.  The leaving key takes
    // the same R_K loads: k~_col = serial fmaf chain over ascending j from +0, which with 8 warps the
    // first half runs over rows 0..63 and the second continues over rows 64..127 from that value
    float acck = 0.f;
    {
        const int col = c & (kD - 1), hf = c / kD;
        constexpr int kRows = kPrepWarps == 8 ? kD / 2 : kD;
        float acc[G];
#pragma unroll
        for (int i = 0; i < G; ++i) acc[i] = 0.f;
        const float* R = p.rk + (size_t)h * kD * kD + col;
        const int jb = hf * kRows;
        for (int j0 = jb; j0 < jb + kRows; j0 += 32) {
            float r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __ldg(R + (size_t)(j0 + j) * kD);
#pragma unroll
            for (int j = 0; j < 32; ++j)
#pragma unroll
                for (int i = 0; i < G; ++i) acc[i] = fmaf(qs[i][j0 + j], r[j], acc[i]);
            if (evict && hf == 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) acck = __fmaf_rn(xk[j0 + j], r[j], acck);
            }
        }
        if constexpr (kPrepWarps == 8) {
            // the output partials' space is free until the BF16 part: the second half's sums, then
            // the key's chain value at row 64
            float* part2 = &ow[0][0][0];
            if (hf == 1) {
#pragma unroll
                for (int i = 0; i < G; ++i) part2[i * kD + col] = acc[i];
            } else if (evict) {
                part2[G * kD + col] = acck;
            }
            __syncthreads();
            if (hf == 0) {
#pragma unroll
                for (int i = 0; i < G; ++i) p.qrot[qbase + (size_t)i * kD + col] = acc[i] + part2[i * kD + col];
            } else if (evict) {
                float k2 = part2[G * kD + col];
#pragma unroll 8
                for (int j = kD / 2; j < kD; ++j) k2 = __fmaf_rn(xk[j], __ldg(R + (size_t)j * kD), k2);
                part2[G * kD + col] = k2;
            }
            // the partial sums are read before this barrier and the key's value right after it, ahead of
            // store_token's barriers: all before any warp writes its output partial into this space
            __syncthreads();
            if (evict) acck = part2[G * kD + (c & (kD - 1))];
        } else {
#pragma unroll
            for (int i = 0; i < G; ++i) p.qrot[qbase + (size_t)i * kD + col] = acc[i];
        }
    }
    if (evict) {
        // clip, quantise and pack the leaving token into its INT2 slot (threads c < 128 hold
        // channel c; thread c >= 128 of an 8-warp CTA only takes part in the barriers)
        const AppendReq& r = ap->req[b];
        const int pg = (r.e0 - kSink) / kPage;
        const int phys = ap->page_table[(size_t)b * ap->max_pps + pg];
        uint8_t* blk = ap->pool + ((size_t)phys * p.hkv + h) * ap->fmt.bytes;
        tq::store_token(blk, ap->fmt, (r.e0 - kSink) % kPage, c < kD ? acck : 0.f, yv, ap->clip_k, ap->clip_v, red,
                        tpart, ap->vmax + (size_t)b * p.hkv + h);
    }

    // ---- BF16 sink + window
    // causal view (chunked prefill): head row x of query token x / g_real sees positions <= lim + x / g_real;
    // a window slot holds position w0 + ((slot - 64 - (w0 - 64)) mod 256), w0 the window's first position
    const int w0 = max(kSink, len - kWindow);
    const int lim = p.lim[b];
    auto slot_pos = [&](int sl) { return sl < kSink ? sl : w0 + (((sl - kSink) - (w0 - kSink)) % kWindow + kWindow) % kWindow; };
    // query fragments: k-step ks holds channels 16 ks + 2 tig + e (+ 8 for registers 2, 3);
    // row g = bf16 high part of head g + 8 k, row g + 8 = its bf16 low part
    uint32_t qa[MT][8][4];
#pragma unroll
    for (int k = 0; k < MT; ++k) {
        const int hd = g + 8 * k;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            float hv[2][2], lv[2][2];
#pragma unroll
            for (int f = 0; f < 2; ++f)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float x = hd < G ? qs[hd][16 * ks + 8 * f + 2 * tig + e] * kQScaleP : 0.f;
                    const float hi = __bfloat162float(__float2bfloat16_rn(x));
                    hv[f][e] = hi;
                    lv[f][e] = x - hi;
                }
            qa[k][ks][0] = pack_bf16x2(hv[0][0], hv[0][1]);
            qa[k][ks][1] = pack_bf16x2(lv[0][0], lv[0][1]);
            qa[k][ks][2] = pack_bf16x2(hv[1][0], hv[1][1]);
            qa[k][ks][3] = pack_bf16x2(lv[1][0], lv[1][1]);
        }
    }
    float m[MT], lpart[MT];           // running max of head g + 8 k (base 2); this thread's part of the sum
#pragma unroll
    for (int k = 0; k < MT; ++k) m[k] = -INFINITY, lpart[k] = 0.f;
    // unnormalised output^T: channel tile cm (channels 16 cm + g, + 8) x heads 8 k + 2 tig, + 1
    float o[8][MT][4];
#pragma unroll
    for (int cm = 0; cm < 8; ++cm)
#pragma unroll
        for (int k = 0; k < MT; ++k) o[cm][k][0] = o[cm][k][1] = o[cm][k][2] = o[cm][k][3] = 0.f;

    for (int i = 0; i < kTiles; ++i) {
        asm volatile("cp.async.wait_group 1;" ::: "memory");   // tile i has landed (tile i + 1 may not)
        __syncwarp();
        const int nt = warp + kPrepWarps * i;
        if (!tile_used(nt)) {   // whole tile empty (or past the region)
            request_tile(i + 2);
            continue;
        }
        const int s0 = 8 * nt;
        const uint8_t* kbuf = wbuf + (i & 1) * kTileBytes;
        const uint8_t* vbuf = kbuf + 8 * kKRow;
        // scores of slots s0 .. s0 + 7
        float acc[MT][4];
#pragma unroll
        for (int k = 0; k < MT; ++k) acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.f;
        const uint8_t* krow = kbuf + g * kKRow + 4 * tig;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(krow + 32 * ks);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(krow + 32 * ks + 16);
#pragma unroll
            for (int k = 0; k < MT; ++k) mma_bf16(acc[k], qa[k][ks], b0, b1);
        }
        // online softmax of head g + 8 k over the tile's slots 2 tig, 2 tig + 1; the probabilities stay
        // in the score layout, which is the B operand of the P.V MMA (k = slot, n = head)
        uint32_t phi[MT], plo[MT];
        float fk[MT];
#pragma unroll
        for (int k = 0; k < MT; ++k) {
            float x[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int sl = s0 + 2 * tig + e;
                const bool seen = lim == INT32_MAX || slot_pos(sl) <= lim + (g + 8 * k) / p.g_real;
                x[e] = slot_live(sl, n_sink, n_win) && seen ? acc[k][e] + acc[k][2 + e] : -INFINITY;
            }
            float cm = fmaxf(x[0], x[1]);
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 1));
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 2));
            const float mn = fmaxf(m[k], cm);
            // mn is -inf only while a row (under the causal view of chunked prefill) has seen no slot
            const bool none = mn == -INFINITY;
            const float f = none ? 1.f : (m[k] == -INFINITY ? 0.f : exp2_approx(m[k] - mn));
            const float p0 = none ? 0.f : exp2_approx(x[0] - mn), p1 = none ? 0.f : exp2_approx(x[1] - mn);
            lpart[k] = fmaf(lpart[k], f, p0 + p1);
            m[k] = mn;
            fk[k] = f;
            // p = high + low part in bf16 (about 16 significant bits)
            const float h0 = __bfloat162float(__float2bfloat16_rn(p0)), h1 = __bfloat162float(__float2bfloat16_rn(p1));
            phi[k] = pack_bf16x2(h0, h1);
            plo[k] = pack_bf16x2(p0 - h0, p1 - h1);
        }
        // value rows of slots outside the sink and window may hold any bits (NaN included), which an MMA
        // with P = 0 would still carry into the output: zero them first.  A tile lies wholly in the sink
        // or wholly in the window region, so its live slots are one run from its first slot
        if (!slot_live(s0 + 7, n_sink, n_win)) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int idx = lane + 32 * q, t = idx >> 4, piece = idx & 15;
                if (!slot_live(s0 + t, n_sink, n_win))
                    *reinterpret_cast<uint4*>(const_cast<uint8_t*>(vbuf) + kKRow * t + 16 * piece) = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }
        // rescale the output columns (heads 8 k + 2 tig + e; their factors sit in row groups 2 tig + e)
#pragma unroll
        for (int k = 0; k < MT; ++k) {
            const float f0 = __shfl_sync(0xffffffffu, fk[k], (2 * tig) * 4);
            const float f1 = __shfl_sync(0xffffffffu, fk[k], (2 * tig + 1) * 4);
#pragma unroll
            for (int cm = 0; cm < 8; ++cm) {
                o[cm][k][0] *= f0;
                o[cm][k][1] *= f1;
                o[cm][k][2] *= f0;
                o[cm][k][3] *= f1;
            }
        }
        // P.V on the tensor cores: O^T += V^T P^T, A = V^T of 16 channels (ldmatrix, transposed),
        // B = P high and low parts
        const uint32_t vaddr = ptx::smem_u32(vbuf) + kKRow * (lane & 7) + 16 * (lane >> 3);
#pragma unroll
        for (int cp = 0; cp < 4; ++cp) {
            uint32_t a[4];
            ldmatrix_x4_trans(a, vaddr + 64 * cp);
#pragma unroll
            for (int k = 0; k < MT; ++k) {
                mma_bf16_k8(o[2 * cp][k], a[0], a[1], phi[k]);
                mma_bf16_k8(o[2 * cp][k], a[0], a[1], plo[k]);
                mma_bf16_k8(o[2 * cp + 1][k], a[2], a[3], phi[k]);
                mma_bf16_k8(o[2 * cp + 1][k], a[2], a[3], plo[k]);
            }
        }
        __syncwarp();            // every lane is done with buffer i & 1 before it is refilled
        request_tile(i + 2);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");

    // ---- merge the warps' partials and write this request's BF16 partial
#pragma unroll
    for (int k = 0; k < MT; ++k) {
        float l = lpart[k];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const int hd = g + 8 * k;
        if (tig == 0 && hd < G) {
            mw[warp][hd] = m[k];
            lw[warp][hd] = l;
        }
    }
#pragma unroll
    for (int cm = 0; cm < 8; ++cm)
#pragma unroll
        for (int k = 0; k < MT; ++k)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int hd = 8 * k + 2 * tig + e;
                if (hd < G) {
                    ow[warp][hd][16 * cm + g] = o[cm][k][e];
                    ow[warp][hd][16 * cm + g + 8] = o[cm][k][2 + e];
                }
            }
    __syncthreads();
    float* part = p.part_bf16 + ((size_t)b * p.hkv + h) * G * (2 + kD);
    const int col = c & (kD - 1);
    for (int i = c / kD; i < G; i += NT / kD) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kPrepWarps; ++w) M = fmaxf(M, mw[w][i]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kPrepWarps; ++w) {
                const float f = mw[w][i] == -INFINITY ? 0.f : exp2_approx(mw[w][i] - M);
                L = fmaf(f, lw[w][i], L);
                O = fmaf(f, ow[w][i][col], O);
            }
        }
        float* ph = part + (size_t)i * (2 + kD);
        if (col == 0) {
            ph[0] = M;
            ph[1] = L;
        }
        ph[2 + col] = O;
    }
}

template <int G>
__global__ void __launch_bounds__(32 * prep_warps(G)) prep(const __grid_constant__ DecodeParams p) {
    prep_body<G, false>(p, nullptr);
}

template <int G>
__global__ void __launch_bounds__(32 * prep_warps(G)) prep_step(const __grid_constant__ DecodeParams p,
                                                                 const __grid_constant__ AppendParams a) {
    prep_body<G, true>(p, &a);
}

// Launch with the per-warp tile buffers as dynamic shared memory (opted in once per device).
template <int G, bool STEP>
cudaError_t launch_prep_g(const DecodeParams& p, const AppendParams* a, cudaStream_t s) {
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        if constexpr (STEP)
            e = cudaFuncSetAttribute(prep_step<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, prep_dyn_smem(G));
        else
            e = cudaFuncSetAttribute(prep<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, prep_dyn_smem(G));
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    const dim3 grid(p.hkv, p.batch);
    if constexpr (STEP)
        prep_step<G><<<grid, 32 * prep_warps(G), prep_dyn_smem(G), s>>>(p, *a);
    else
        prep<G><<<grid, 32 * prep_warps(G), prep_dyn_smem(G), s>>>(p);
    return cudaGetLastError();
}

template <bool STEP>
cudaError_t launch_prep_any(const DecodeParams& p, const AppendParams* a, cudaStream_t s) {
    switch (p.g) {
        case 1: return launch_prep_g<1, STEP>(p, a, s);
        case 2: return launch_prep_g<2, STEP>(p, a, s);
        case 3: return launch_prep_g<3, STEP>(p, a, s);
        case 4: return launch_prep_g<4, STEP>(p, a, s);
        case 5: return launch_prep_g<5, STEP>(p, a, s);
        case 6: return launch_prep_g<6, STEP>(p, a, s);
        case 7: return launch_prep_g<7, STEP>(p, a, s);
        case 8: return launch_prep_g<8, STEP>(p, a, s);
        case 12: return launch_prep_g<12, STEP>(p, a, s);
        case 16: return launch_prep_g<16, STEP>(p, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_prep_step(const DecodeParams& p, const AppendParams& a, cudaStream_t s) {
    return launch_prep_any<true>(p, &a, s);
}

cudaError_t launch_prep(const DecodeParams& p, cudaStream_t s) {
    return launch_prep_any<false>(p, nullptr, s);
}

}  // namespace oscar
