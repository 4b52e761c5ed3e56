// append.cu -- write path of the INT2 rotated paged KV cache (sm_103a).
//
// kv_quant_append runs two kernels on the caller's stream:
//   1. quant_few (decode steps: at most 8 tokens per page and head) or quant_pages (prefill,
//      chunked appends): one CTA per (touched INT2 page, KV head).  Every position that
//      leaves the BF16 window in this call (or goes straight to INT2 in a long
//      append) is rotated (keys only), clipped, quantised to asymmetric INT2 in two
//      64-channel groups and packed into its page (axbrief.com OSCAR page, section
//      "attention-statistics rotation + Triton kernels": k . R_K, c_K = 0.96,
//      c_V = 0.92, G_K = 64, per-token asymmetric INT2; values unrotated because R_V
//      is folded into W_V / W_O offline).
//   2. insert_bf16: copies the new tokens that stay in BF16 into the sink / window
//      slots and publishes the new lengths (axbrief.com OSCAR page, section "OSCAR
//      release": BF16 sink + recent window).
// Stream order makes kernel 1 read the window before kernel 2 overwrites it.  A decode step made
// through oscar_decode_step does the same work for its one token per request inside prep_step
// (prep.cu) with the per-token quantisation of token_quant.h, which quant_few uses as well.
// kv_quant_append_layers runs the same two kernels once for all layers of a model (the *_layers
// forms: one parameter block per layer in device memory, the layer in blockIdx.z).  Every writer
// also raises the (request, KV head)'s recorded largest value scale (AppendParams::vmax).
//
// Bit-exact contract (shared with nothing but the written specification): the key
// rotation is the serial chain acc = fma(x_j, R[j][c], acc), j = 0..127, acc0 = +0;
// clip products, the range subtraction and the divisions are single IEEE fp32
// operations (explicit _rn intrinsics, so the compiler cannot contract them);
// fp16 conversions round to nearest even; codes are rint (ties to even) of the IEEE
// quotient, decided by the equivalent exact compares of token_quant.h.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "token_quant.h"

namespace oscar {
namespace {

using namespace tq;

__device__ __forceinline__ int find_request(const AppendParams& p, int job) {
    int b = 0;
    for (int i = 1; i < p.batch; ++i)
        if (p.req[i].e1 > p.req[i].e0 && p.req[i].job0 <= job) b = i;
    return b;
}

constexpr int kFew = 8;   // tokens per (page, KV head) up to which quant_few is used

// Appends that quantise at most kFew tokens per (page, KV head) -- every decode step: thread =
// channel, the kFew tokens' rotation chains side by side, block-wide group min / max per token.
__device__ __forceinline__ void quant_few_body(const AppendParams& p, const int job, const int h) {
    extern __shared__ __align__(16) float smem[];
    float* R = smem;                   // [128][128]
    float* xs = R + kD * kD;           // [kFew][128]
    float* red = xs + kFew * kD;       // [8]
    __shared__ uint8_t part[2][4][16];  // [K|V][warp][lane < 16]: half-packed code bytes of one token

    const int c = threadIdx.x;
    const int b = find_request(p, job);
    const AppendReq& r = p.req[b];
    const int pg = r.page0 + (job - r.job0);
    const int pbeg = max(r.e0, kSink + pg * kPage);
    const int pend = min(r.e1, kSink + (pg + 1) * kPage);
    const int phys = p.page_table[(size_t)b * p.max_pps + pg];
    uint8_t* blk = p.pool + ((size_t)phys * p.hkv + h) * p.fmt.bytes;

    {   // stage R_K of this head with asynchronous 16-byte copies, all of a thread's 32 in flight
        // at once (waited for before the first __syncthreads below)
        const float4* src = reinterpret_cast<const float4*>(p.rk + (size_t)h * kD * kD);
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(R);
#pragma unroll
        for (int i = 0; i < kD * kD / 4 / 128; ++i)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16u * (c + 128 * i)),
                         "l"(src + c + 128 * i)
                         : "memory");
    }
    for (int p0 = pbeg; p0 < pend; p0 += kFew) {
        const int n = min(kFew, pend - p0);
        __syncthreads();
        for (int t = 0; t < n; ++t) xs[t * kD + c] = bf16_bits_to_f32(token_src(p, b, h, 0, p0 + t)[c]);
        if (p0 == pbeg) asm volatile("cp.async.wait_all;" ::: "memory");   // R_K has landed
        __syncthreads();
        // keys: k~_c = sum_j x_j R[j][c], serial fused multiply-add in ascending j (one chain per
        // token; a decode step brings one token per (page, KV head), which takes the single chain)
        float acc[kFew];
#pragma unroll
        for (int t = 0; t < kFew; ++t) acc[t] = 0.0f;
        if (n == 1) {
#pragma unroll 8
            for (int j = 0; j < kD; ++j) acc[0] = __fmaf_rn(xs[j], R[j * kD + c], acc[0]);
        } else {
#pragma unroll 4
            for (int j = 0; j < kD; ++j) {
                const float rj = R[j * kD + c];
#pragma unroll
                for (int t = 0; t < kFew; ++t) acc[t] = __fmaf_rn(xs[t * kD + j], rj, acc[t]);
            }
        }
        for (int t = 0; t < n; ++t) {
            // K (rotated) and V (unrotated): per-token asymmetric INT2 in two 64-channel groups
            const float yv = bf16_bits_to_f32(token_src(p, b, h, 1, p0 + t)[c]);
            store_token(blk, p.fmt, (p0 + t - kSink) % kPage, acc[t], yv, p.clip_k, p.clip_v, red, part,
                        p.vmax + (size_t)b * p.hkv + h);
        }
    }
}

// OR of a value over the four lanes whose channel blocks differ in bits 1..2 (code position r)
__device__ __forceinline__ uint32_t or_over_r(uint32_t v) {
    v |= __shfl_xor_sync(0xffffffffu, v, 2);
    v |= __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}

// min / max over the lanes of a group: 8 lanes for 64 channels (channel blocks differing in bits
// 0..2), 16 lanes for 128 channels (bits 0..3)
__device__ __forceinline__ GroupStat group_minmax_lanes(float mn, float mx, int group) {
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (group == kD) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    }
    GroupStat g;
    g.mn = mn;
    g.mx = mx;
    return g;
}

constexpr int kQPThreads = 256;   // threads of quant_pages

// Position of float4 f (channels 4f .. 4f + 3) inside a staged R_K row: bit 0 flipped when bit 3 is
// set.  Thread cb reads float4s 2 cb and 2 cb + 1; unswizzled, the 16 lanes of a token would fall
// on only 4 of the 8 bank groups of a 128-byte row (4-way conflicts), swizzled they cover all 8.
__device__ __forceinline__ int rk_swz(int f) { return f ^ ((f >> 3) & 1); }
constexpr int kSPT = kPage * 16 / kQPThreads;   // page slots per thread (16 lanes per slot)

// One CTA per (touched INT2 page, KV head), 256 threads.  Thread t owns the 4 page slots
// 4 (t >> 4) .. + 3 and the 8 channels 8 cb .. 8 cb + 7 (cb = t & 15), so a token's 128 channels sit
// in 16 lanes of one warp and a 64-channel group in 8 of them: group min / max and the packing of
// four codes per byte are warp shuffles, with no block-wide barrier per token.
// Keys: the 64 x 128 tile times R_K with each output the serial fmaf chain over ascending j
// (the bit-exact contract), 4 tokens x 8 channels of independent chains per thread.
__device__ __forceinline__ void quant_pages_body(const AppendParams& p, const int job, const int h) {
    extern __shared__ __align__(16) float smem[];
    float* R = smem;                   // [128][128]
    float* xt = R + kD * kD;           // [128][64]: key inputs, channel-major (xt[j][slot]); after the
                                       // rotation, the page-head block being built (full pages)
    uint16_t* vt = reinterpret_cast<uint16_t*>(xt + kD * kPage);   // [64][128]: value rows (bf16)

    const int t = threadIdx.x;
    const int tb = t >> 4, cb = t & 15;
    const int b = find_request(p, job);
    const AppendReq& r = p.req[b];
    const int pg = r.page0 + (job - r.job0);
    const int page_pos = kSink + pg * kPage;                 // position of slot 0
    const int pbeg = max(r.e0, page_pos);
    const int pend = min(r.e1, page_pos + kPage);
    const int sbeg = pbeg - page_pos, send = pend - page_pos;
    const int phys = p.page_table[(size_t)b * p.max_pps + pg];
    uint8_t* blk = p.pool + ((size_t)phys * p.hkv + h) * p.fmt.bytes;

    {   // stage R_K of this head (asynchronous 16-byte copies, all in flight while the key inputs
        // of the page's live slots are loaded) and those key inputs.  Row j keeps its 32 float4s
        // with the index swizzled (rk_swz), so that the rotation's row loads hit every bank
        const float4* src = reinterpret_cast<const float4*>(p.rk + (size_t)h * kD * kD);
        const uint32_t dst = (uint32_t)__cvta_generic_to_shared(R);
#pragma unroll
        for (int i = 0; i < kD * kD / 4 / kQPThreads; ++i) {
            const int idx = t + kQPThreads * i, row = idx >> 5, f = idx & 31;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16u * (32 * row + rk_swz(f))),
                         "l"(src + idx)
                         : "memory");
        }
        // value rows of the live slots, also asynchronous (read by the quantisation below)
        const uint32_t vdst = (uint32_t)__cvta_generic_to_shared(vt);
#pragma unroll
        for (int i = 0; i < kPage * (kD / 8) / kQPThreads; ++i) {
            const int idx = t + kQPThreads * i, s = idx >> 4, ch = 8 * (idx & 15);
            if (s >= sbeg && s < send)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(vdst + 2u * (s * kD + ch)),
                             "l"(token_src(p, b, h, 1, page_pos + s) + ch)
                             : "memory");
        }
        // key inputs: 16-byte loads (8 channels of one token), 8 independent ones per thread; the 32
        // lanes of a warp take 32 slots of one channel block, so the transposed stores hit 32 banks
        for (int idx = t; idx < kPage * (kD / 8); idx += kQPThreads) {
            const int s = idx & (kPage - 1), ch = 8 * (idx >> 6);
            if (s < sbeg || s >= send) continue;
            const uint4 w = *reinterpret_cast<const uint4*>(token_src(p, b, h, 0, page_pos + s) + ch);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                xt[(ch + 2 * k) * kPage + s] = bf16_bits_to_f32((uint16_t)(ws[k] & 0xffff));
                xt[(ch + 2 * k + 1) * kPage + s] = bf16_bits_to_f32((uint16_t)(ws[k] >> 16));
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    }
    __syncthreads();

    // ---- keys: k~[s][c] = sum_j x[s][j] R[j][c], serial fused multiply-add in ascending j.  Two
    // channels' chains share one packed f32x2 FMA; each lane of it rounds exactly as a scalar fmaf
    float2 acc2[kSPT][4];
#pragma unroll
    for (int i = 0; i < kSPT; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) acc2[i][m] = make_float2(0.0f, 0.0f);
    const int f0 = rk_swz(2 * cb), f1 = rk_swz(2 * cb + 1);
    // 16 steps per loop pass: their shared-memory addresses become immediate offsets (measured: 3.7%
    // faster bulk appends than 2 steps per pass; the fully unrolled loop was no faster than 2)
#pragma unroll 16
    for (int j = 0; j < kD; ++j) {
        const float4 x0 = *reinterpret_cast<const float4*>(xt + j * kPage + kSPT * tb);
        const float4 r0 = reinterpret_cast<const float4*>(R + j * kD)[f0];
        const float4 r1 = reinterpret_cast<const float4*>(R + j * kD)[f1];
        const float xv[kSPT] = {x0.x, x0.y, x0.z, x0.w};
        const float2 rv[4] = {make_float2(r0.x, r0.y), make_float2(r0.z, r0.w), make_float2(r1.x, r1.y),
                              make_float2(r1.z, r1.w)};
#pragma unroll
        for (int i = 0; i < kSPT; ++i)
#pragma unroll
            for (int m = 0; m < 4; ++m) acc2[i][m] = __ffma2_rn(make_float2(xv[i], xv[i]), rv[m], acc2[i][m]);
    }
    float acc[kSPT][8];
#pragma unroll
    for (int i = 0; i < kSPT; ++i)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            acc[i][2 * m] = acc2[i][m].x;
            acc[i][2 * m + 1] = acc2[i][m].y;
        }
    // a page filled completely by this call is built in shared memory (in the key-input space, free
    // now) and written out with 16-byte stores; a partly filled one is updated byte by byte in place
    const bool whole = sbeg == 0 && send == kPage;
    uint8_t* ob = whole ? reinterpret_cast<uint8_t*>(xt) : blk;
    __syncthreads();

    // ---- per token: clip, quantise, pack.  Channel c = 8 cb + jj: group u = cb >> 3, code
    // position r = (cb >> 1) & 3, y = cb & 1 in both page orders.
    const int u = cb >> 3, rpos = (cb >> 1) & 3, y = cb & 1;
    uint32_t vbig = 0;   // largest fp16 value scale (bits) of this thread's live tokens
#pragma unroll
    for (int i = 0; i < kSPT; ++i) {
        const int s = kSPT * tb + i;
        const bool live = s >= sbeg && s < send;      // same for the 16 lanes of the token
        if (!__any_sync(0xffffffffu, live)) continue;
        // keys
        {
            float mn = acc[i][0], mx = acc[i][0];
#pragma unroll
            for (int jj = 1; jj < 8; ++jj) mn = fminf(mn, acc[i][jj]), mx = fmaxf(mx, acc[i][jj]);
            const GroupStat gs = group_minmax_lanes(mn, mx, p.fmt.gk);
            // code of channel 8 cb + jj at bits 2 rpos of byte jj & 3 of word jj >> 2; after the OR
            // over the four code positions every byte is complete
            uint32_t w[2] = {0u, 0u};
            const QuantGroup qg = quant_group(gs, p.clip_k);
            const uint16_t s16 = qg.s16, m16 = qg.m16;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                w[jj >> 2] |= (uint32_t)quant_code(acc[i][jj], qg) << (8 * (jj & 3) + 2 * rpos);
            w[0] = or_over_r(w[0]);
            w[1] = or_over_r(w[1]);
            // the row's word at 8 x + 4 u holds the bytes (e, y) = (0, 0), (0, 1), (1, 0), (1, 1) of
            // channels 2 x + e: the y = 0 lane writes x = 0, 1 and the y = 1 lane x = 2, 3
            const uint32_t p0 = __shfl_xor_sync(0xffffffffu, w[0], 1), p1 = __shfl_xor_sync(0xffffffffu, w[1], 1);
            if (live && rpos == 0) {
                const uint32_t lo = y ? p1 : w[0], hi = y ? w[1] : p0;   // bytes of lane y = 0 / y = 1
                uint8_t* row = ob + kKCodes + s * 32 + 16 * y + 4 * u;
                *reinterpret_cast<uint32_t*>(row) = __byte_perm(lo, hi, 0x5140);
                *reinterpret_cast<uint32_t*>(row + 8) = __byte_perm(lo, hi, 0x7362);
            }
            if (live && (8 * cb) % p.fmt.gk == 0)
                *reinterpret_cast<uint32_t*>(ob + p.fmt.k_sm + s * p.fmt.k_stride + (8 * cb / p.fmt.gk) * 4) =
                    (uint32_t)s16 | ((uint32_t)m16 << 16);
        }
        // values (unrotated): this thread's 8 channels of the token, straight from the source row
        {
            float vx[8];
            if (live) {
                const uint4 w = *reinterpret_cast<const uint4*>(vt + s * kD + 8 * cb);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    vx[2 * k] = bf16_bits_to_f32((uint16_t)(ws[k] & 0xffff));
                    vx[2 * k + 1] = bf16_bits_to_f32((uint16_t)(ws[k] >> 16));
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) vx[k] = 0.f;
            }
            float mn = vx[0], mx = vx[0];
#pragma unroll
            for (int jj = 1; jj < 8; ++jj) mn = fminf(mn, vx[jj]), mx = fmaxf(mx, vx[jj]);
            const GroupStat gs = group_minmax_lanes(mn, mx, p.fmt.gv);
            uint32_t w[2] = {0u, 0u};
            const QuantGroup qg = quant_group(gs, p.clip_v);
            const uint16_t s16 = qg.s16, m16 = qg.m16;
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                w[jj >> 2] |= (uint32_t)quant_code(vx[jj], qg) << (8 * (jj & 3) + 2 * rpos);
            w[0] = or_over_r(w[0]);
            w[1] = or_over_r(w[1]);
            // channel 8 cb + jj = 64 u + 16 rpos + 8 y + jj: the byte of (slot s, channel 64 u + 8 y + jj)
            if (live && rpos == 0) {
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    ob[p.fmt.v_codes + v_code_byte(s, 64 * u + 8 * y + jj)] = (uint8_t)(w[jj >> 2] >> (8 * (jj & 3)));
            }
            if (live && (8 * cb) % p.fmt.gv == 0)
                *reinterpret_cast<uint32_t*>(ob + p.fmt.v_sm + s * p.fmt.v_stride + (8 * cb / p.fmt.gv) * 4) =
                    (uint32_t)s16 | ((uint32_t)m16 << 16);
            if (live) vbig = max(vbig, (uint32_t)s16);
        }
    }
    vbig = __reduce_max_sync(0xffffffffu, vbig);
    if ((t & 31) == 0 && vbig) atomicMax(p.vmax + (size_t)b * p.hkv + h, vbig);
    if (whole) {
        __syncthreads();
        for (int i = t; i < p.fmt.bytes / 16; i += kQPThreads)
            reinterpret_cast<uint4*>(blk)[i] = reinterpret_cast<const uint4*>(ob)[i];
    }
}

// New tokens that stay in BF16 (sink, or the final window) -> their slots.  One CTA per (request, KV
// head, K or V); the rows are copied as 16-byte pieces, all independent, so a CTA keeps many loads
// in flight instead of one row at a time.
constexpr int kInsThreads = 256;
__device__ __forceinline__ void insert_bf16_body(const AppendParams& p, const int b, const int h, const int kv) {
    const AppendReq& r = p.req[b];
    const int l1 = r.len0 + r.n_new;
    const int wstart = max(kSink, l1 - kWindow);
    // sink positions [len0, min(l1, sink)), then the final window [max(len0, wstart), l1): disjoint
    const int a0 = r.len0, n0 = max(0, min(l1, kSink) - r.len0);
    const int a1 = max(r.len0, wstart), n1 = max(0, l1 - a1);
    const uint4* src = reinterpret_cast<const uint4*>(kv == 0 ? p.k : p.v);
    uint4* dst = reinterpret_cast<uint4*>(p.bf16 + (((size_t)b * p.hkv + h) * 2 + kv) * kSlots * kD);
    constexpr int kPieces = kD * 2 / 16;   // 16-byte pieces per 128-channel bf16 row
    const int total = (n0 + n1) * kPieces;
#pragma unroll 4
    for (int idx = threadIdx.x; idx < total; idx += kInsThreads) {
        const int row = idx / kPieces, piece = idx - row * kPieces;
        const int pos = row < n0 ? a0 + row : a1 + (row - n0);
        const uint4 w = __ldg(src + ((size_t)(r.tok_off + (pos - r.len0)) * p.hkv + h) * kPieces + piece);
        dst[(size_t)bf16_slot(pos) * kPieces + piece] = w;
    }
    if (h == 0 && kv == 0 && threadIdx.x == 0) p.seq_lens[b] = l1;
}

// Kernels.  One cache: the parameters are a kernel argument.  Several layers in one launch: one
// parameter block per layer in device memory, the layer in blockIdx.z (blockIdx.z / 2 for the window
// insert, whose z also selects K or V).
__global__ void __launch_bounds__(128) quant_few(const __grid_constant__ AppendParams p) {
    quant_few_body(p, blockIdx.x, blockIdx.y);
}
__global__ void __launch_bounds__(128) quant_few_layers(const AppendParams* __restrict__ ps) {
    quant_few_body(ps[blockIdx.z], blockIdx.x, blockIdx.y);
}
__global__ void __launch_bounds__(kQPThreads) quant_pages(const __grid_constant__ AppendParams p) {
    quant_pages_body(p, blockIdx.x, blockIdx.y);
}
__global__ void __launch_bounds__(kQPThreads) quant_pages_layers(const AppendParams* __restrict__ ps) {
    quant_pages_body(ps[blockIdx.z], blockIdx.x, blockIdx.y);
}
__global__ void __launch_bounds__(kInsThreads) insert_bf16(const __grid_constant__ AppendParams p) {
    insert_bf16_body(p, blockIdx.x, blockIdx.y, blockIdx.z);
}
__global__ void __launch_bounds__(kInsThreads) insert_bf16_layers(const AppendParams* __restrict__ ps) {
    insert_bf16_body(ps[blockIdx.z >> 1], blockIdx.x, blockIdx.y, blockIdx.z & 1);
}

constexpr size_t kSmemTiled = (size_t)(kD * kD + kD * kPage) * sizeof(float) + (size_t)kPage * kD * sizeof(uint16_t);
constexpr size_t kSmemFew = (size_t)(kD * kD + kFew * kD + 8) * sizeof(float);

// dynamic shared-memory opt-in of the quantisation kernels, once per device
cudaError_t append_attrs() {
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(quant_pages, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTiled);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(quant_pages_layers, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTiled);
        if (e == cudaSuccess) e = cudaFuncSetAttribute(quant_few, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemFew);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(quant_few_layers, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemFew);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return cudaSuccess;
}

// at most kFew tokens leave the window per request (every decode step): the per-channel kernel;
// otherwise (prefill, chunked appends) the tiled one
bool few_tokens(const AppendParams& p) {
    int most = 0;
    for (int b = 0; b < p.batch; ++b) most = max(most, p.req[b].e1 - p.req[b].e0);
    return most <= kFew;
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t s) {
    cudaError_t e = append_attrs();
    if (e != cudaSuccess) return e;
    int n = 0;
    if (p.n_jobs > 0) {
        if (few_tokens(p))
            quant_few<<<dim3(p.n_jobs, p.hkv), 128, kSmemFew, s>>>(p);
        else
            quant_pages<<<dim3(p.n_jobs, p.hkv), kQPThreads, kSmemTiled, s>>>(p);
        ++n;
    }
    insert_bf16<<<dim3(p.batch, p.hkv, 2), kInsThreads, 0, s>>>(p);
    ++n;
    count_launches(n);
    return cudaGetLastError();
}

cudaError_t launch_append_layers(const AppendParams* dev_params, const AppendParams& p0, int n_layers, cudaStream_t s) {
    cudaError_t e = append_attrs();
    if (e != cudaSuccess) return e;
    int n = 0;
    if (p0.n_jobs > 0) {
        if (few_tokens(p0))
            quant_few_layers<<<dim3(p0.n_jobs, p0.hkv, n_layers), 128, kSmemFew, s>>>(dev_params);
        else
            quant_pages_layers<<<dim3(p0.n_jobs, p0.hkv, n_layers), kQPThreads, kSmemTiled, s>>>(dev_params);
        ++n;
    }
    insert_bf16_layers<<<dim3(p0.batch, p0.hkv, 2 * n_layers), kInsThreads, 0, s>>>(dev_params);
    ++n;
    count_launches(n);
    return cudaGetLastError();
}

}  // namespace oscar
