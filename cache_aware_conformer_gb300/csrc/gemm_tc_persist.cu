// Persistent tcgen05 GEMM for problems with many output tiles (the offline
// encode, M in the thousands): C = A * B^T with the fused epilogues of gemm.cuh.
//
// 128 x 128 output tiles; one CTA per SM walks tiles t = blockIdx.x,
// blockIdx.x + gridDim.x, ... (tile t = row block t / (N / 128), column block
// t % (N / 128), so neighbouring CTAs share A rows in L2).  Two TMEM
// accumulators (2 x 128 fp32 columns) let the epilogue of one tile run while
// the main loop fills the other:
//   warp 0 lane 0  TMA producer: one continuous STAGES-deep ring over all the
//                  CTA's tiles and K slices (A as a plain or split (hi, lo)
//                  operand, or the convolution view of a window buffer);
//   warp 1 lane 0  MMA issuer: per tile, waits for a free accumulator, issues
//                  4 (split: 8) tcgen05.mma per 64-wide K slice, releases each
//                  slice with tcgen05.commit and signals the full accumulator;
//   warps 2-5      epilogue warpgroup: warp w reads TMEM lanes 32 (w % 4) ..
//                  (one output row per thread, 32-column chunks), applies the
//                  fused epilogue, then frees the accumulator.
// Every mbarrier wait is bounded; a wait that gives up latches CAC_E_TIMEOUT
// and the CTA unwinds.
#include "gemm.cuh"

namespace cac {

namespace {
constexpr int PBM = 128, PBN = 128, PBK = 64;
constexpr int P_THREADS = 192;
constexpr int P_A_TILE = PBM * PBK * 2;
constexpr int P_B_TILE = PBN * PBK * 2;

template <int SPLIT>
struct PCfg {
    static constexpr int A_TILES = P_A_TILE * (1 + SPLIT);
    static constexpr int STAGE = A_TILES + P_B_TILE;
    static constexpr int STAGES = SPLIT ? 4 : 6;
    static constexpr int SMEM = STAGES * STAGE + 1024 /*align slack*/ + 256 /*barriers*/;
    static_assert(SMEM <= 227 * 1024, "shared memory");
};
}  // namespace

template <int KIND, int SPLIT>
__global__ void __launch_bounds__(P_THREADS, 1)
    gemm_tc_persist_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M,
                           int N, int K, int conv_C, EpiParams ep, int* status) {
    using C = PCfg<SPLIT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_TILES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::STAGES * P_B_TILE);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;  // [2] accumulator ready for the epilogue
    uint64_t* tempty = tfull + 2;         // [2] accumulator drained by the epilogue
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles_n = N / PBN, tiles = ((M + PBM - 1) / PBM) * tiles_n;
    const int nk = K / PBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);  // one arrival per epilogue warp
        }
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 2 * PBN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();

    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
                const int m0 = (t / tiles_n) * PBM, n0 = (t % tiles_n) * PBN;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % C::STAGES;
                    if (it >= C::STAGES && !mbar_wait(&empty[s], ((it / C::STAGES) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    const int k0 = kb * PBK;
                    mbar_expect_tx(&full[s], C::STAGE);
                    tma_load_2d(sB + s * P_B_TILE, &tmB, k0, n0, &full[s]);
                    uint8_t* a = sA + s * C::A_TILES;
                    if (conv_C) {
                        const int tap = k0 / conv_C;
                        tma_load_3d(a, &tmA, k0 - tap * conv_C, tap & 1, m0 + (tap >> 1), &full[s]);
                        if (SPLIT)
                            tma_load_3d(a + P_A_TILE, &tmA, conv_C + k0 - tap * conv_C, tap & 1, m0 + (tap >> 1),
                                        &full[s]);
                    } else {
                        tma_load_2d(a, &tmA, k0, m0, &full[s]);
                        if (SPLIT) tma_load_2d(a + P_A_TILE, &tmA, K + k0, m0, &full[s]);
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(PBM, PBN);
            int it = 0, lt = 0;
            for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x, ++lt) {
                const int acc = lt & 1;
                if (!mbar_wait(&tempty[acc], ((lt >> 1) & 1) ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * PBN);
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = it % C::STAGES;
                    if (!mbar_wait(&full[s], (it / C::STAGES) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sdesc_k_sw128(sA + s * C::A_TILES);
                    const uint64_t bd = sdesc_k_sw128(sB + s * P_B_TILE);
#pragma unroll
                    for (int kk = 0; kk < PBK / 16; ++kk) tc_mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
                    if (SPLIT) {
                        const uint64_t al = sdesc_k_sw128(sA + s * C::A_TILES + P_A_TILE);
#pragma unroll
                        for (int kk = 0; kk < PBK / 16; ++kk) tc_mma_bf16(d, al + 2 * kk, bd + 2 * kk, idesc, 1u);
                    }
                    tc_commit(&empty[s]);
                }
                tc_commit(&tfull[acc]);
            }
        }
    } else {
        // epilogue warpgroup (warps 2..5: TMEM lane quarters 2, 3, 0, 1)
        const int quarter = warp & 3;
        int lt = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++lt) {
            const int acc = lt & 1;
            if (!mbar_wait(&tfull[acc], (lt >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int m0 = (t / tiles_n) * PBM, n0 = (t % tiles_n) * PBN;
            const int row = m0 + quarter * 32 + lane;
#pragma unroll 1
            for (int c = 0; c < PBN; c += 32) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * PBN + c), v);
                if (row < M) {
                    EpiPre pre;
                    epi_prefetch<KIND>(ep, row, n0 + c, pre);
                    epilogue32<KIND, bf16>(ep, row, n0 + c, v, pre);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
        }
    }
    pdl_trigger();
    if (!ok) latch_error(status, CAC_E_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 2 * PBN);
}

template <int KIND, int SPLIT>
static cudaError_t launch_p(const CUtensorMap* tmA, const CUtensorMap* tmB, int M, int N, int K, int conv_C,
                            const EpiParams& ep, int* status, cudaStream_t s) {
    using C = PCfg<SPLIT>;
    auto kern = gemm_tc_persist_kernel<KIND, SPLIT>;
    static bool attr_set = false;
    static int sms = 0;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        attr_set = true;
    }
    const int tiles = ((M + PBM - 1) / PBM) * (N / PBN);
    return launch_k(kern, dim3(std::min(tiles, sms)), dim3(P_THREADS), C::SMEM, s, 1, *tmA, *tmB, M, N, K, conv_C,
                    ep, status);
}

cudaError_t launch_gemm_tc_persistent(const CUtensorMap* tmA, const CUtensorMap* tmB128, int M, int N, int K,
                                      int conv_C, int a_split, const EpiParams& ep, int* status, cudaStream_t s) {
    if (M <= 0) return cudaSuccess;
    if (K % PBK || K <= 0 || N % PBN || !ep.act_bf16) return cudaErrorInvalidValue;
    if (conv_C && (conv_C % PBK || K != 3 * conv_C)) return cudaErrorInvalidValue;
    if (a_split) {
        switch (ep.kind) {
            case EPI_STORE: return launch_p<EPI_STORE, 1>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
            case EPI_RESID: return launch_p<EPI_RESID, 1>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
            case EPI_GLU: return launch_p<EPI_GLU, 1>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
            case EPI_QKV: return launch_p<EPI_QKV, 1>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
            case EPI_SUB: return launch_p<EPI_SUB, 1>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (ep.kind) {
        case EPI_STORE: return launch_p<EPI_STORE, 0>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
        case EPI_RESID: return launch_p<EPI_RESID, 0>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
        case EPI_GLU: return launch_p<EPI_GLU, 0>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
        case EPI_QKV: return launch_p<EPI_QKV, 0>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
        case EPI_SUB: return launch_p<EPI_SUB, 0>(tmA, tmB128, M, N, K, conv_C, ep, status, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace cac
