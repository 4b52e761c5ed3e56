// calib.cu -- offline calibration of the key rotation R_K = U_Q * H_Had * P_br (sm_103a).
//
// axbrief.com OSCAR page, section "attention-statistics rotation + Triton kernels": U_Q are
// the eigenvectors of the query covariance C_Q = (1/N) sum_n q_n^T q_n; H_Had is the
// normalised Hadamard transform and P_br the bit-reversal permutation (techllm.github.io
// page, section "OSCAR": they spread important channels evenly).
//
// Three kernels per call, one CTA per KV head for the eigen-solver:
//   covariance   C = (1/n) Q^T Q in fp64.
//   jacobi       parallel cyclic Jacobi (round-robin ordering: 64 disjoint rotations per
//                round, 127 rounds per sweep) on C held in shared memory, accumulating the
//                eigenvectors in global memory; sweeps until the off-diagonal Frobenius
//                norm is <= 1e-15 * ||C||_F (at most 40 sweeps).
//   assemble     sort eigenpairs by descending eigenvalue, sign each eigenvector so its
//                largest-magnitude entry is positive, R[r][c] = sum_k U[r][k] H[k][brev(c)],
//                H[k][i] = (-1)^popcount(k & i) / sqrt(128); rounded to fp32.
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

cudaError_t launch_build_rk(const float* q, int64_t n, int hkv, float* rk, void* ws, cudaStream_t s) {
    double* w = (double*)ws;
    covariance<<<dim3(kN, hkv), 128, 0, s>>>(q, n, w);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int smem = kN * kN * sizeof(double);
    e = cudaFuncSetAttribute(jacobi, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    jacobi<<<hkv, 1024, smem, s>>>(w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    assemble<<<hkv, 128, 0, s>>>(w, rk);
    count_launches(3);
    return cudaGetLastError();
}

}  // namespace oscar
