// internal.h -- shared definitions of the CUDA kernels and the host side of the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

struct oscar_cache;

namespace oscar {

constexpr int kD = 128;            // head_dim
constexpr int kPage = 64;          // INT2 tokens per page
constexpr int kGroup = 64;         // channels per quantisation group
constexpr int kSink = 64;          // BF16 sink tokens
constexpr int kWindow = 256;       // BF16 recent-window tokens
constexpr int kSlots = kSink + kWindow;
constexpr int kMaxBatch = 256;     // requests per call (kernel-parameter tables)
constexpr int kMaxAppendLayers = 4096;   // caches per kv_quant_append_layers call (grid z = 2 x layers)
constexpr int kMaxG = 16;          // query heads per KV head
constexpr int kMaxDevices = 64;    // devices whose per-device launch settings are cached

// Byte layout of one (physical page, KV head) block with 64-channel groups for keys and values
// (the largest format; PageFmt below gives the layout for every group-size pair).
constexpr int kKCodes = 0;                      // [64 tokens][32 B] key codes (k_code_byte / k_code_shift)
constexpr int kKSm = 2048;                      // [64 tokens][s0 m0 s1 m1] fp16
constexpr int kVCodes = 2560;                   // 2048 B of value codes (v_code_byte / v_code_shift)
constexpr int kVSm = 4608;                      // [64 tokens][s0 m0 s1 m1] fp16
constexpr int kPageHeadBytes = 5120;

// Layout of a (page, KV head) block when keys are quantised in groups of gk channels and values in
// groups of gv channels (64 or 128 each): key codes, key scale/min (one fp16 pair per group and
// token), value codes, value scale/min.  The code regions are the same for every format.
struct PageFmt {
    int32_t gk, gv;                 // channels per quantisation group: keys, values
    int32_t k_stride, v_stride;     // scale/min bytes per token: 4 * (128 / group)
    int32_t k_sm, v_codes, v_sm;    // byte offsets of the key scale/min, value codes, value scale/min
    int32_t bytes;                  // bytes of the block (a multiple of 16)
};
__host__ __device__ inline PageFmt page_fmt(int gk, int gv) {
    PageFmt f;
    f.gk = gk;
    f.gv = gv;
    f.k_stride = 4 * (kD / gk);
    f.v_stride = 4 * (kD / gv);
    f.k_sm = 2048;
    f.v_codes = f.k_sm + kPage * f.k_stride;
    f.v_sm = f.v_codes + 2048;
    f.bytes = f.v_sm + kPage * f.v_stride;
    return f;
}

// Where the 2-bit codes sit inside a page.  The order is chosen for the warp-level MMA read
// path: each thread of a warp finds the codes of its mma.m16n8k16 fragments in one 8-byte
// (keys) or 16-byte (values) shared-memory load, and every fragment register comes out of a
// word with one AND (codes land in fp16 subnormals code * 4^r * 2^-24, r = k_code_shift / 2).
//   keys, token row t (32 B): channel c = 64u + 16r + 8y + 2x + e  ->  byte 8x + 4u + 2e + y, bits 2r
//   values: token t = 32a + 16k + 8s + 2x + e, channel c = 64q + 16r + 8y + g
//           ->  byte 1024a + 512q + 16(4g + x) + 4(2k + s) + 2e + y of the value region, bits 2r
__host__ __device__ inline int k_code_byte(int c) {
    return 8 * ((c >> 1) & 3) + 4 * (c >> 6) + 2 * (c & 1) + ((c >> 3) & 1);
}
__host__ __device__ inline int k_code_shift(int c) { return 2 * ((c >> 4) & 3); }
__host__ __device__ inline int v_code_byte(int t, int c) {
    return 1024 * (t >> 5) + 512 * (c >> 6) + 16 * (4 * (c & 7) + ((t >> 1) & 3)) + 4 * (2 * ((t >> 4) & 1) + ((t >> 3) & 1)) +
           2 * (t & 1) + ((c >> 3) & 1);
}
__host__ __device__ inline int v_code_shift(int c) { return 2 * ((c >> 4) & 3); }

// Slot of position p in the BF16 region of one (request, KV head, K|V).
__host__ __device__ inline int bf16_slot(int64_t p) {
    return p < kSink ? (int)p : kSink + (int)((p - kSink) % kWindow);
}

struct AppendReq {
    int32_t len0;     // tokens before this call
    int32_t n_new;    // tokens appended by this call
    int64_t tok_off;  // first row of this request in the k / v input
    int32_t e0, e1;   // INT2 positions quantised by this call: [e0, e1)
    int32_t job0;     // index of this request's first page job
    int32_t page0;    // logical INT2 page of e0
};

struct AppendParams {
    PageFmt fmt;
    int32_t batch, hkv, n_jobs;
    float clip_k, clip_v;
    const uint16_t* k;     // bf16 [rows][hkv][128]
    const uint16_t* v;
    const float* rk;       // [hkv][128][128]
    uint8_t* pool;
    uint16_t* bf16;        // [batch][hkv][2][kSlots][128]
    const int32_t* page_table;
    int32_t* seq_lens;
    int32_t max_pps;
    uint32_t* vmax;        // [batch][hkv] largest fp16 value scale quantised so far (fp16 bits)
    AppendReq req[kMaxBatch];
};

struct DecodeParams {
    PageFmt fmt;
    int32_t batch, hkv, g, pps, max_splits;
    const void* q;
    int32_t q_dtype;
    const float* rk;
    void* out;
    int32_t out_dtype;
    const uint8_t* pool;
    const uint16_t* bf16;
    const int32_t* page_table;
    int32_t max_pps;
    float* qrot;           // [batch][hkv*g][128]
    float* partial;        // SIMT path: [batch][hkv][max_splits][g][2 + 128]
    int32_t len[kMaxBatch];
    int32_t path;          // OSCAR_PATH_SIMT (1) or OSCAR_PATH_WARP_MMA (2)
    float* part_mma;       // warp-MMA path: [batch * hkv + n_units][g][2 + 128], slot (b * hkv + h) + unit
    float* part_bf16;      // [batch * hkv][g][2 + 128]: the BF16 sink / window split
    int32_t* err;          // nonzero after a bounded wait gave up
    const uint32_t* vmax;  // [batch][hkv] largest fp16 value scale in the request's INT2 pages (bits)
    int32_t wait_iters;    // a bounded wait gives up after this many tests of up to 1 ms each
    int32_t wait_probe;    // nonzero: the first kernel also waits on a barrier nothing arrives at
    // warp-MMA path
    int32_t total_pages;   // INT2 pages over all (request, KV head)
    int32_t n_units;       // page-streaming units (warps) of the warp-MMA kernel
    int32_t page_off[kMaxBatch + 1];   // sum over earlier requests of pages * hkv
    // Request slots and query rows.  Slot b of a launch reads the page-table row, BF16 region and
    // cached tokens of request row[b] (len[b] is that request's length); its g query rows are qpr
    // query tokens x g_real heads, query j of the slot being row q0[b] + j of the caller's q and out
    // ([rows][hkv * g_real][128]) and seeing positions <= lim[b] + j; rows of queries j >= nq[b] are
    // unused.  A decode call is the identity (row[b] = q0[b] = b, qpr = 1, nq = 1, lim = INT32_MAX);
    // chunked prefill packs qpr queries of one request into a slot.
    int32_t g_real, qpr;
    int32_t row[kMaxBatch];
    int32_t q0[kMaxBatch];
    int32_t nq[kMaxBatch];
    int32_t lim[kMaxBatch];
};

// The per-request metadata buffer (seq_lens) holds the lengths, int32[batch], then from this byte
// offset the largest fp16 value scale quantised so far per (request, KV head), uint32[batch][hkv]
// (fp16 bits; a positive fp16 value orders like its bits).  The read path takes its fp16 range
// limit for P' = p * s_V from it once per (request, KV head) instead of testing every page.
__host__ __device__ inline size_t vmax_offset(int batch) { return ((size_t)batch * 4 + 15) / 16 * 16; }

// Split-K partition of one request: INT2 splits of `pps` pages plus one BF16 split.
__host__ __device__ inline int int2_tokens(int len) {
    return len > kSlots ? len - kSlots : 0;
}
__host__ __device__ inline int int2_pages(int len) {
    return (int2_tokens(len) + kPage - 1) / kPage;
}
__host__ __device__ inline int int2_splits(int len, int pps) {
    return (int2_pages(len) + pps - 1) / pps;
}

constexpr int kMaxMmaUnits = 2048;     // units of one warp-MMA launch (partial-buffer slots)

// Launchers (each returns the cudaError_t of its launch).
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
// The same for several caches (layers) that append the same tokens per request: parameter blocks in
// device memory (dev_params[layer]); p0 is layer 0's host copy (grid sizes, kernel choice).
cudaError_t launch_append_layers(const AppendParams* dev_params, const AppendParams& p0, int n_layers, cudaStream_t s);
// timing: null, or two events recorded on `s` around the INT2 attention kernel's launch
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s, cudaEvent_t* timing = nullptr);
cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t s);
// the transposed-score kernel (decode_mma_t.cu) for the head counts it serves: G <= 4 and G = 12
bool decode_mma_t_serves(int g);
int mma_t_units_per_cta(int g);   // warps per CTA of the transposed-score kernel
cudaError_t launch_decode_mma_t(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_prep(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_prep_step(const DecodeParams& p, const AppendParams& a, cudaStream_t s);
// fused decode step (warp-MMA path): prep with the append of one token per request, then the INT2
// attention and the combine
cudaError_t launch_decode_step(const DecodeParams& p, const AppendParams& a, cudaStream_t s,
                               cudaEvent_t* timing = nullptr);
int mma_units_per_cta(int g);   // warps per CTA of the warp-MMA decode kernel that serves G heads per KV head
cudaError_t launch_build_rk(const float* q, int64_t n, int hkv, float* rk, void* ws, cudaStream_t s);
size_t build_rk_ws_bytes(int hkv);
size_t cq_acc_bytes(int hkv);
cudaError_t launch_cq_accumulate(const float* q, int64_t n, int hkv, void* acc, cudaStream_t s);
cudaError_t launch_cq_finalize(const void* acc, int hkv, float* rk, void* ws, cudaStream_t s);
int sv_max_keys();
cudaError_t launch_score_weighted(const float* q, int64_t n, const float* k, const float* v, int t_keys, int hkv, float* y,
                                  cudaStream_t s);

void count_launches(int n);

// Byte offset of the error word inside the fixed scratch of oscar_decode_attention_noalloc.
constexpr size_t kNoallocErrOffset = 0;

// Parameters of a warp-MMA decode using one fixed scratch buffer (see noalloc.cu).
int noalloc_decode_params(oscar_cache* c, const void* q, int32_t q_dtype, const float* rk, void* out,
                          int32_t out_dtype, void* scratch, size_t scratch_bytes, DecodeParams* p,
                          cudaStream_t stream);

}  // namespace oscar
