// token_quant.h -- per-token INT2 quantisation of one key / value vector, thread = channel, shared
// by the write-path kernels and the fused decode step (device code only).
//
// The arithmetic is the write path's bit-exact contract (axbrief.com OSCAR page, section
// "attention-statistics rotation + Triton kernels": per-token asymmetric INT2 in 64-channel groups
// (128-channel groups as a per-cache option, the variants behind the page's 2.28 / 2.38 bits),
// c_K = 0.96, c_V = 0.92): clip products, the range subtraction and the division by 3 are single
// IEEE fp32 operations (explicit _rn intrinsics), fp16 conversions round to nearest even, and each
// code is the one rint of the IEEE quotient (x - m) / s gives, decided by exact compares (quant_code).
#pragma once

#include <cuda_fp16.h>

#include "internal.h"

namespace oscar {
namespace tq {

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

// Source row (bf16[128]) of position `pos` of request b, KV head h, tensor kv (0 = K, 1 = V).
__device__ __forceinline__ const uint16_t* token_src(const AppendParams& p, int b, int h, int kv,
                                                     int pos) {
    const AppendReq& r = p.req[b];
    if (pos < r.len0) {   // still in the BF16 window (it leaves it in this call)
        size_t base = (((size_t)b * p.hkv + h) * 2 + kv) * kSlots + bf16_slot(pos);
        return p.bf16 + base * kD;
    }
    const uint16_t* t = kv == 0 ? p.k : p.v;
    return t + ((size_t)(r.tok_off + (pos - r.len0)) * p.hkv + h) * kD;
}

struct GroupStat {
    float mn, mx;
};

struct Quant {
    int code;
    uint16_t s16, m16;
};

// What one group's codes depend on: the clip range, the fp16 minimum m and the three code
// thresholds of the fp16 scale s.
struct QuantGroup {
    float lo, hi, m;
    float t0, t1, t2;
    uint16_t s16, m16;
};

// The code of a value is clamp(rint(fl((xc - m) / s)), 0, 3) with one IEEE division and
// round-half-even.  Because s is an fp16 value (at most 11 significant bits), 0.5 s, 1.5 s and 2.5 s
// are exact fp32 numbers, and the halfway points of the division (0.5 + 2^-25, 1.5 - 2^-24 and
// 2.5 + 2^-23 times s) each fall strictly inside one fp32 spacing of them.  So, for d = fl(xc - m),
//   rint(fl(d / s)) >= 1  iff  d >  0.5 s     (rint(0.5) = 0)
//   rint(fl(d / s)) >= 2  iff  d >= 1.5 s     (rint(1.5) = 2)
//   rint(fl(d / s)) >= 3  iff  d >  2.5 s     (rint(2.5) = 2)
// and the code is the number of thresholds d passes: the same code, decided by three compares
// instead of a division per value.  s = 0 gives code 0 (all thresholds +inf).
__device__ __forceinline__ QuantGroup quant_group(GroupStat g, float clip) {
    QuantGroup q;
    q.lo = __fmul_rn(clip, g.mn);
    q.hi = __fmul_rn(clip, g.mx);
    const float s_exact = __fdiv_rn(__fsub_rn(q.hi, q.lo), 3.0f);
    q.s16 = __half_as_ushort(__float2half_rn(s_exact));
    q.m16 = __half_as_ushort(__float2half_rn(q.lo));
    const float s = __half2float(__ushort_as_half(q.s16));
    q.m = __half2float(__ushort_as_half(q.m16));
    const bool zero = s == 0.0f;
    q.t0 = zero ? INFINITY : __fmul_rn(0.5f, s);
    q.t1 = zero ? INFINITY : __fmul_rn(1.5f, s);
    q.t2 = zero ? INFINITY : __fmul_rn(2.5f, s);
    return q;
}

__device__ __forceinline__ int quant_code(float y, const QuantGroup& q) {
    const float d = __fsub_rn(fminf(fmaxf(y, q.lo), q.hi), q.m);
    return (int)(d > q.t0) + (int)(d >= q.t1) + (int)(d > q.t2);
}

__device__ __forceinline__ Quant quantise(float y, GroupStat g, float clip) {
    const QuantGroup qg = quant_group(g, clip);
    Quant q;
    q.code = quant_code(y, qg);
    q.s16 = qg.s16;
    q.m16 = qg.m16;
    return q;
}

// Min and max over the channels of each group: threads 0..63 and 64..127 for 64-channel groups,
// threads 0..127 for one 128-channel group.
__device__ __forceinline__ GroupStat group_minmax(float y, float* red, int group) {
    float mn = y, mx = y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[2 * w] = mn;
        red[2 * w + 1] = mx;
    }
    __syncthreads();
    GroupStat g;
    if (group == kD) {
        g.mn = fminf(fminf(red[0], red[2]), fminf(red[4], red[6]));
        g.mx = fmaxf(fmaxf(red[1], red[3]), fmaxf(red[5], red[7]));
    } else {
        const int w0 = (w & 3) & ~1;
        g.mn = fminf(red[2 * w0], red[2 * w0 + 2]);
        g.mx = fmaxf(red[2 * w0 + 1], red[2 * w0 + 3]);
    }
    __syncthreads();
    return g;
}

// Quantise one token (channel c of the key y_k and value y_v in thread c < 128; any further threads
// of the block take part in the barriers only) and store its codes and scales into slot `slot` of the
// page-head block `blk` (layout f).  `red` holds 2 floats per warp of the block, `part` 2 x 4 x 16 bytes.
// The value scales also raise *vmax, the largest fp16 value scale of the (request, KV head).
__device__ __forceinline__ void store_token(uint8_t* blk, const PageFmt& f, int slot, float yk, float yv, float clip_k,
                                            float clip_v, float* red, uint8_t (*part)[4][16], uint32_t* vmax) {
    const int c = threadIdx.x, lane = c & 31;
    const Quant qk = quantise(yk, group_minmax(yk, red, f.gk), clip_k);
    const Quant qv = quantise(yv, group_minmax(yv, red, f.gv), clip_v);
    if (c < kD && (c & (f.gk - 1)) == 0)
        *reinterpret_cast<uint32_t*>(blk + f.k_sm + slot * f.k_stride + (c / f.gk) * 4) =
            (uint32_t)qk.s16 | ((uint32_t)qk.m16 << 16);
    if (c < kD && (c & (f.gv - 1)) == 0) {
        *reinterpret_cast<uint32_t*>(blk + f.v_sm + slot * f.v_stride + (c / f.gv) * 4) =
            (uint32_t)qv.s16 | ((uint32_t)qv.m16 << 16);
        if (qv.s16) atomicMax(vmax, (uint32_t)qv.s16);
    }
    // pack: every code byte holds the codes of four channels c0 + 16 r (r = 0..3) of this token, two
    // from lanes l and l ^ 16 of one warp and two from the next warp
    uint32_t pk = (uint32_t)qk.code << k_code_shift(c & (kD - 1));
    uint32_t pv = (uint32_t)qv.code << v_code_shift(c & (kD - 1));
    pk |= __shfl_xor_sync(0xffffffffu, pk, 16);
    pv |= __shfl_xor_sync(0xffffffffu, pv, 16);
    if (c < kD && lane < 16) {
        part[0][c >> 5][lane] = (uint8_t)pk;
        part[1][c >> 5][lane] = (uint8_t)pv;
    }
    __syncthreads();
    if (c < 32) {
        // key byte c of the token row: channels 64u + 16r + 8y + 2x + e
        const int x = c >> 3, u = (c >> 2) & 1, e = (c >> 1) & 1, y = c & 1;
        const int l = 8 * y + 2 * x + e;
        blk[kKCodes + slot * 32 + c] = part[0][2 * u][l] | part[0][2 * u + 1][l];
    } else if (c < 64) {
        // value byte of channels 64q + 16r + 8y + g
        const int j = c - 32, q = j >> 4, g = (j >> 1) & 7, y = j & 1;
        const int l = 8 * y + g;
        blk[f.v_codes + v_code_byte(slot, 64 * q + 8 * y + g)] = part[1][2 * q][l] | part[1][2 * q + 1][l];
    }
    __syncthreads();   // part and red are free again
}

}  // namespace tq
}  // namespace oscar
