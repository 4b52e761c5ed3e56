// calib.cu -- offline calibration of the key rotation R_K = U_Q * H_Had * P_br (sm_103a).
//
// axbrief.com OSCAR page, section "attention-statistics rotation + Triton kernels": U_Q are
// the eigenvectors of the query covariance C_Q = (1/N) sum_n q_n^T q_n; H_Had is the
// normalised Hadamard transform and P_br the bit-reversal permutation (techllm.github.io
// page, section "OSCAR": they spread important channels evenly).
//
// Three kernels per call, one CTA per KV head for the eigen-solver:
//   covariance   C = (1/n) Q^T Q in fp64 (or, streaming over several calls, cq_accumulate adds
//                sum_t q_t^T q_t and the sample count into a caller-owned accumulator and
//                cq_normalise divides once at the end).
//   jacobi       parallel cyclic Jacobi (round-robin ordering: 64 disjoint rotations per
//                round, 127 rounds per sweep) on C held in shared memory, accumulating the
//                eigenvectors in global memory; sweeps until the off-diagonal Frobenius
//                norm is <= 1e-15 * ||C||_F (at most 40 sweeps).
//   assemble     sort eigenpairs by descending eigenvalue, sign each eigenvector so its
//                largest-magnitude entry is positive, R[r][c] = sum_k U[r][k] H[k][brev(c)],
//                H[k][i] = (-1)^popcount(k & i) / sqrt(128); rounded to fp32.
// score_weighted computes the calibration samples of the value rotation: rows of S V, whose
// covariance is C_S = (1/N) V^T S^T S V (same page and section); R_V is then built from them by
// the same eigen-solver and assembly.
#include "internal.h"

namespace oscar {
namespace {

constexpr int kN = kD;

__global__ void __launch_bounds__(128) covariance(const float* __restrict__ q, int64_t n,
                                                  double* __restrict__ ws) {
    const int h = blockIdx.y;
    const int i = blockIdx.x;
    const int j = threadIdx.x;
    const float* qh = q + (size_t)h * n * kN;
    double acc = 0.0;
    for (int64_t t = 0; t < n; ++t) acc = fma((double)qh[t * kN + i], (double)qh[t * kN + j], acc);
    ws[(size_t)h * 2 * kN * kN + (size_t)i * kN + j] = acc / (double)n;
}

// Streaming form of the covariance: sums[h][i][j] += sum_t q_ti q_tj over this call's samples (fp64,
// every sample in order, so a run of calls adds the same products a single call would), and
// counts[h] += n.
__global__ void __launch_bounds__(128) cq_accumulate(const float* __restrict__ q, int64_t n, double* __restrict__ sums,
                                                     long long* __restrict__ counts) {
    const int h = blockIdx.y;
    const int i = blockIdx.x;
    const int j = threadIdx.x;
    const float* qh = q + (size_t)h * n * kN;
    double acc = 0.0;
    for (int64_t t = 0; t < n; ++t) acc = fma((double)qh[t * kN + i], (double)qh[t * kN + j], acc);
    sums[(size_t)h * kN * kN + (size_t)i * kN + j] += acc;
    if (i == 0 && j == 0) counts[h] += (long long)n;
}

// C = sums / count into the eigen-solver's workspace (the layout the covariance kernel writes)
__global__ void __launch_bounds__(128) cq_normalise(const double* __restrict__ sums, const long long* __restrict__ counts,
                                                    double* __restrict__ ws) {
    const int h = blockIdx.y;
    const int i = blockIdx.x;
    const int j = threadIdx.x;
    const double c = (double)counts[h];
    ws[(size_t)h * 2 * kN * kN + (size_t)i * kN + j] = sums[(size_t)h * kN * kN + (size_t)i * kN + j] / c;
}

// Rows of S V for calibration: y_i = sum_t softmax_t(q_i . k_t / sqrt(128)) v_t for every query i of
// every head h (one CTA per (query, head), thread = channel).  Logits in fp32 (four warps, one key
// each, lanes over channels), each probability exp(logit - max) once in fp32, the sums of p and of
// p v in fp64.
constexpr int kSvMaxKeys = 8192;
__global__ void __launch_bounds__(128) score_weighted(const float* __restrict__ q, int64_t n, const float* __restrict__ k,
                                                      const float* __restrict__ v, int t_keys, float* __restrict__ y) {
    extern __shared__ float lg[];     // [t_keys]
    __shared__ float qs[kN];
    __shared__ float red[4];
    __shared__ double dred[4];
    const int h = blockIdx.y;
    const int64_t i = blockIdx.x;
    const int c = threadIdx.x, w = c >> 5, lane = c & 31;
    qs[c] = q[((size_t)h * n + i) * kN + c];
    __syncthreads();
    const float* kh = k + (size_t)h * t_keys * kN;
    const float* vh = v + (size_t)h * t_keys * kN;
    const float scale = 0.08838834764831845f;   // 1 / sqrt(128)
    float mx = -INFINITY;
    for (int t = w; t < t_keys; t += 4) {
        const float4 kv = *reinterpret_cast<const float4*>(kh + (size_t)t * kN + 4 * lane);
        float d = qs[4 * lane] * kv.x;
        d = fmaf(qs[4 * lane + 1], kv.y, d);
        d = fmaf(qs[4 * lane + 2], kv.z, d);
        d = fmaf(qs[4 * lane + 3], kv.w, d);
        for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
        d *= scale;
        if (lane == 0) lg[t] = d;
        mx = fmaxf(mx, d);
    }
    if (lane == 0) red[w] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    // probabilities (unnormalised), each computed once, in place of the logits
    double lp = 0.0;
    for (int t = c; t < t_keys; t += kN) {
        const float pr = expf(lg[t] - mx);
        lg[t] = pr;
        lp += (double)pr;
    }
    for (int o = 16; o > 0; o >>= 1) lp += __shfl_xor_sync(0xffffffffu, lp, o);
    if (lane == 0) dred[w] = lp;
    __syncthreads();
    const double l = (dred[0] + dred[1]) + (dred[2] + dred[3]);
    double acc = 0.0;
    for (int t = 0; t < t_keys; ++t) acc = fma((double)lg[t], (double)vh[(size_t)t * kN + c], acc);
    y[((size_t)h * n + i) * kN + c] = (float)(acc / l);
}

__device__ __forceinline__ int rr_player(int slot, int round) {
    // circle method: slot 0 is fixed, the other 127 rotate
    return slot == 0 ? 0 : 1 + (slot - 1 + round) % (kN - 1);
}

__global__ void __launch_bounds__(1024) jacobi(double* __restrict__ ws) {
    extern __shared__ __align__(16) double a[];   // [128][128]
    __shared__ double cs[kN / 2], sn[kN / 2];
    __shared__ int pp[kN / 2], qq[kN / 2];
    __shared__ double red[32];
    __shared__ int done;
    const int h = blockIdx.x;
    const int tid = threadIdx.x;
    double* cg = ws + (size_t)h * 2 * kN * kN;
    double* v = cg + kN * kN;
    for (int i = tid; i < kN * kN; i += blockDim.x) {
        a[i] = cg[i];
        v[i] = (i / kN == i % kN) ? 1.0 : 0.0;
    }
    __syncthreads();
    // ||A||_F
    double f = 0.0;
    for (int i = tid; i < kN * kN; i += blockDim.x) f += a[i] * a[i];
    for (int o = 16; o > 0; o >>= 1) f += __shfl_xor_sync(0xffffffffu, f, o);
    if ((tid & 31) == 0) red[tid >> 5] = f;
    __syncthreads();
    double fro = 0.0;
    for (int w = 0; w < 32; ++w) fro += red[w];
    fro = sqrt(fro);
    __syncthreads();

    for (int sweep = 0; sweep < 40; ++sweep) {
        double off = 0.0;
        for (int i = tid; i < kN * kN; i += blockDim.x)
            if (i / kN != i % kN) off += a[i] * a[i];
        for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
        if ((tid & 31) == 0) red[tid >> 5] = off;
        __syncthreads();
        if (tid == 0) {
            double s = 0.0;
            for (int w = 0; w < 32; ++w) s += red[w];
            done = sqrt(s) <= 1e-15 * fro;
        }
        __syncthreads();
        if (done) break;
        for (int round = 0; round < kN - 1; ++round) {
            if (tid < kN / 2) {
                int x = rr_player(tid, round), y = rr_player(kN - 1 - tid, round);
                int p = min(x, y), q = max(x, y);
                pp[tid] = p;
                qq[tid] = q;
                double apq = a[p * kN + q];
                double c = 1.0, s = 0.0;
                if (apq != 0.0) {
                    double tau = (a[q * kN + q] - a[p * kN + p]) / (2.0 * apq);
                    double t = (tau >= 0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
                    c = 1.0 / sqrt(1.0 + t * t);
                    s = t * c;
                }
                cs[tid] = c;
                sn[tid] = s;
            }
            __syncthreads();
            // rows: A <- J^T A
            for (int task = tid; task < (kN / 2) * kN; task += blockDim.x) {
                int k = task / kN, col = task % kN;
                int p = pp[k], q = qq[k];
                double c = cs[k], s = sn[k];
                double ap = a[p * kN + col], aq = a[q * kN + col];
                a[p * kN + col] = c * ap - s * aq;
                a[q * kN + col] = s * ap + c * aq;
            }
            __syncthreads();
            // columns: A <- A J, and V <- V J
            for (int task = tid; task < (kN / 2) * kN; task += blockDim.x) {
                int k = task % (kN / 2), row = task / (kN / 2);
                int p = pp[k], q = qq[k];
                double c = cs[k], s = sn[k];
                double ap = a[row * kN + p], aq = a[row * kN + q];
                a[row * kN + p] = c * ap - s * aq;
                a[row * kN + q] = s * ap + c * aq;
                double vp = v[row * kN + p], vq = v[row * kN + q];
                v[row * kN + p] = c * vp - s * vq;
                v[row * kN + q] = s * vp + c * vq;
            }
            __syncthreads();
        }
    }
    // eigenvalues back to global (first row of the C area is reused as scratch)
    if (tid < kN) cg[tid] = a[tid * kN + tid];
}

__device__ __forceinline__ int brev7(int i) { return __brev((unsigned)i) >> 25; }

__global__ void __launch_bounds__(128) assemble(const double* __restrict__ ws, float* __restrict__ rk) {
    __shared__ int src[kN];
    __shared__ double sg[kN];
    __shared__ double ev[kN];
    const int h = blockIdx.x;
    const int t = threadIdx.x;
    const double* cg = ws + (size_t)h * 2 * kN * kN;
    const double* v = cg + kN * kN;
    ev[t] = cg[t];
    __syncthreads();
    // rank of eigenvalue t in descending order (ties by index)
    int rank = 0;
    for (int j = 0; j < kN; ++j) rank += (ev[j] > ev[t]) || (ev[j] == ev[t] && j < t);
    src[rank] = t;
    __syncthreads();
    {   // sign of output column `t`: largest |entry| positive (first index on ties)
        const int col = src[t];
        int imax = 0;
        double vmax = fabs(v[col]);
        for (int i = 1; i < kN; ++i) {
            double x = fabs(v[i * kN + col]);
            if (x > vmax) {
                vmax = x;
                imax = i;
            }
        }
        sg[t] = v[imax * kN + col] < 0 ? -1.0 : 1.0;
    }
    __syncthreads();
    const double hs = 1.0 / sqrt((double)kN);
    for (int r = 0; r < kN; ++r) {
        // R[r][t] = sum_k U[r][k] H[k][brev(t)], U[r][k] = sg[k] v[r][src[k]]
        const int i = brev7(t);
        double acc = 0.0;
        for (int k = 0; k < kN; ++k) {
            const double u = sg[k] * v[r * kN + src[k]];
            acc += (__popc(k & i) & 1) ? -u : u;
        }
        rk[(size_t)h * kN * kN + r * kN + t] = (float)(acc * hs);
    }
}

}  // namespace

size_t build_rk_ws_bytes(int hkv) { return (size_t)hkv * 2 * kN * kN * sizeof(double); }

// eigen-decomposition of the covariances in ws and the R assembly
static cudaError_t eigen_and_assemble(int hkv, float* rk, double* w, cudaStream_t s) {
    const int smem = kN * kN * sizeof(double);
    cudaError_t e = cudaFuncSetAttribute(jacobi, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    jacobi<<<hkv, 1024, smem, s>>>(w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    assemble<<<hkv, 128, 0, s>>>(w, rk);
    count_launches(2);
    return cudaGetLastError();
}

cudaError_t launch_build_rk(const float* q, int64_t n, int hkv, float* rk, void* ws, cudaStream_t s) {
    double* w = (double*)ws;
    covariance<<<dim3(kN, hkv), 128, 0, s>>>(q, n, w);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
    return eigen_and_assemble(hkv, rk, w, s);
}

size_t cq_acc_bytes(int hkv) { return (size_t)hkv * (kN * kN * sizeof(double) + sizeof(long long)); }

cudaError_t launch_cq_accumulate(const float* q, int64_t n, int hkv, void* acc, cudaStream_t s) {
    double* sums = (double*)acc;
    long long* counts = (long long*)(sums + (size_t)hkv * kN * kN);
    cq_accumulate<<<dim3(kN, hkv), 128, 0, s>>>(q, n, sums, counts);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_cq_finalize(const void* acc, int hkv, float* rk, void* ws, cudaStream_t s) {
    const double* sums = (const double*)acc;
    const long long* counts = (const long long*)(sums + (size_t)hkv * kN * kN);
    double* w = (double*)ws;
    cq_normalise<<<dim3(kN, hkv), 128, 0, s>>>(sums, counts, w);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    count_launches(1);
    return eigen_and_assemble(hkv, rk, w, s);
}

int sv_max_keys() { return kSvMaxKeys; }

cudaError_t launch_score_weighted(const float* q, int64_t n, const float* k, const float* v, int t_keys, int hkv, float* y,
                                  cudaStream_t s) {
    const int smem = t_keys * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(score_weighted, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    score_weighted<<<dim3((unsigned)n, hkv), 128, smem, s>>>(q, n, k, v, t_keys, y);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace oscar
