// SIMT GEMM: C = A * B^T with fp32 FMA on CUDA cores, fp32 or bf16 operands.
// Used for the fp32 mode (tolerance 1e-4 against the fp64 oracle), for the
// load-time position-table product, and as a debugging twin of the tcgen05
// kernel.  64 x 64 output tile per 256-thread CTA, 4 x 4 register micro-tile,
// 16-deep K slices staged through shared memory; the finished tile is staged
// once more in shared memory so the epilogue sees whole 32-column row segments.
#include "gemm.cuh"

namespace cac {

template <class TA, int KIND, class TAct>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const TA* __restrict__ A, long long lda,
                                                        const TA* __restrict__ B, long long ldb, int M, int N,
                                                        int K, int conv_C, int a_split, EpiParams ep) {
    __shared__ float As[16][64 + 4];
    __shared__ float Bs[16][64 + 4];
    __shared__ float Cs[64][64 + 1];
    pdl_trigger();
    pdl_wait();
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = tid * 4 + j, r = e >> 4, kk = e & 15;
            const int gm = m0 + r, gn = n0 + r, gk = k0 + kk;
            float av = 0.f;
            if (gm < M && gk < K) {
                long long off;
                int lo;
                if (conv_C) {
                    const int tap = gk / conv_C;
                    off = (long long)gm * lda + (long long)tap * conv_C * (1 + a_split) + (gk - tap * conv_C);
                    lo = conv_C;
                } else {
                    off = (long long)gm * lda + gk;
                    lo = K;
                }
                av = to_f(A[off]) + (a_split ? to_f(A[off + lo]) : 0.f);
            }
            As[kk][r] = av;
            Bs[kk][r] = (gn < N && gk < K) ? to_f(B[(long long)gn * ldb + gk]) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) { a[i] = As[kk][ty * 4 + i]; b[i] = Bs[kk][tx * 4 + i]; }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) Cs[ty * 4 + i][tx * 4 + j] = acc[i][j];
    __syncthreads();
    if (tid < 128) {
        const int r = tid >> 1, seg = tid & 1;
        const int row = m0 + r, col0 = n0 + 32 * seg;
        if (row < M && col0 < N) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = Cs[r][32 * seg + i];
            EpiPre pre;
            epi_prefetch<KIND>(ep, row, col0, pre);
            epilogue32<KIND, TAct>(ep, row, col0, v, pre);
        }
    }
}

template <class TA, class TAct>
static cudaError_t launch_t(const void* A, long long lda, const void* B, long long ldb, int M, int N, int K,
                           int cc, int sp, const EpiParams& ep, cudaStream_t s) {
    dim3 grid((N + 63) / 64, (M + 63) / 64);
    const TA* a = static_cast<const TA*>(A);
    const TA* b = static_cast<const TA*>(B);
    switch (ep.kind) {
        case EPI_STORE: return launch_k(gemm_simt_kernel<TA, EPI_STORE, TAct>, grid, dim3(256), 0, s, 1, a, lda, b, ldb, M, N, K, cc, sp, ep);
        case EPI_RESID: return launch_k(gemm_simt_kernel<TA, EPI_RESID, TAct>, grid, dim3(256), 0, s, 1, a, lda, b, ldb, M, N, K, cc, sp, ep);
        case EPI_GLU: return launch_k(gemm_simt_kernel<TA, EPI_GLU, TAct>, grid, dim3(256), 0, s, 1, a, lda, b, ldb, M, N, K, cc, sp, ep);
        case EPI_QKV: return launch_k(gemm_simt_kernel<TA, EPI_QKV, TAct>, grid, dim3(256), 0, s, 1, a, lda, b, ldb, M, N, K, cc, sp, ep);
        case EPI_SUB: return launch_k(gemm_simt_kernel<TA, EPI_SUB, TAct>, grid, dim3(256), 0, s, 1, a, lda, b, ldb, M, N, K, cc, sp, ep);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_simt(int bf16_operands, const void* A, long long lda, const void* B, long long ldb, int M,
                             int N, int K, int conv_C, int a_split, const EpiParams& ep, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    if (N % 32 || (conv_C && K != 3 * conv_C)) return cudaErrorInvalidValue;
    if (bf16_operands) return launch_t<bf16, bf16>(A, lda, B, ldb, M, N, K, conv_C, a_split, ep, s);
    if (ep.act_bf16 || a_split) return cudaErrorInvalidValue;
    return launch_t<float, float>(A, lda, B, ldb, M, N, K, conv_C, 0, ep, s);
}

}  // namespace cac
