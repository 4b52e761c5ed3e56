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
constexpr int kMaxG = 16;          // query heads per KV head

// Byte layout of one (physical page, KV head) block.
constexpr int kKCodes = 0;                      // [64 tokens][32 B], channel 4i+j -> byte i bits 2j
constexpr int kKSm = 2048;                      // [64 tokens][s0 m0 s1 m1] fp16
constexpr int kVCodes = 2560;                   // [128 channels][16 B], token 4i+j -> byte i bits 2j
constexpr int kVSm = 4608;                      // [64 tokens][s0 m0 s1 m1] fp16
constexpr int kPageHeadBytes = 5120;

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
    AppendReq req[kMaxBatch];
};

struct DecodeParams {
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
    // tensor-core path
    int32_t path;          // 0 = tensor cores, 1 = SIMT
    int32_t n_cta;         // persistent CTAs
    int32_t total_tiles;   // 128-token INT2 tiles over all (request, KV head)
    float* part_tc;        // [batch * hkv + n_cta][g][2 + 128], segment id = (b * hkv + h) + cta
    float* part_bf16;      // [batch * hkv][g][2 + 128]
    int32_t* err;          // nonzero after a bounded wait gave up
    int32_t tile_off[kMaxBatch + 1];   // sum over earlier requests of tiles * hkv
    // warp-MMA path
    int32_t total_pages;   // INT2 pages over all (request, KV head)
    int32_t n_warps;       // warps of the warp-MMA kernel
    int32_t page_off[kMaxBatch + 1];   // sum over earlier requests of pages * hkv
};

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

constexpr int kTileTok = 128;          // tokens per tensor-core tile (two pages)
constexpr int kMaxCtas = 1024;
__host__ __device__ inline int int2_tiles(int len) {
    return (int2_tokens(len) + kTileTok - 1) / kTileTok;
}

// Launchers (each returns the cudaError_t of its launch).
cudaError_t launch_append(const AppendParams& p, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_tc(const DecodeParams& p, cudaStream_t s);
cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t s);
int mma_warps_per_cta();
cudaError_t launch_build_rk(const float* q, int64_t n, int hkv, float* rk, void* ws, cudaStream_t s);
size_t build_rk_ws_bytes(int hkv);

void count_launches(int n);

// Parameters of a warp-MMA decode using one fixed scratch buffer (see noalloc.cu).
int noalloc_decode_params(oscar_cache* c, const void* q, int32_t q_dtype, const float* rk, void* out,
                          int32_t out_dtype, void* scratch, size_t scratch_bytes, DecodeParams* p,
                          cudaStream_t stream);

}  // namespace oscar
