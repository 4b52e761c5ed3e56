// decode_mma_common.h -- pieces shared by the two warp-MMA INT2 decode kernels (decode_mma.cu: query
// rows as the MMA's A operand; decode_mma_t.cu: key codes as A): the walk over the flattened page
// list, the bounded wait on a page copy, the code-to-fragment conversion, the fp16 MMA and the
// constants of the lazily raised reference maximum (device code only).
#pragma once

#include <cuda_fp16.h>

#include "internal.h"
#include "ptx_async.h"

namespace oscar {
namespace mma_common {

// A raise of the reference max leaves the largest logit this far below tau.  The half step keeps
// the largest probabilities off exact powers of two: with p = 2^k (1 - e) for a nearly flat
// attention, fp16(p * s_V) would round back to the fp16 value 2^k s_V for every token, a bias
// that the output's cancellation between sum P' code and sum p m_V magnifies; at 2^(k + 1/2) the
// rounding errors are spread evenly and average out.
constexpr float kTauSlack = 7.5f;
constexpr float kTauMax = 40.0f;    // tau of a (request, KV head) without a non-zero value scale
constexpr float kQScaleM = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
constexpr float kTwo18 = 262144.0f;

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
    if (ptx::mbar_try(bar, parity)) return true;
    for (int t = 0; t < iters; ++t)
        if (ptx::mbar_try_sleep(bar, parity, 1000000)) return true;
    atomicOr(err, 1);
    return false;
}
constexpr int kDrainIters = 2000;   // copies in flight at a warp's exit: up to about 2 s

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

}  // namespace mma_common
}  // namespace oscar
