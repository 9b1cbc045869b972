// Palette-weight GEMM on the 5th-generation tensor cores: C = A W^T (+ bias),
// A bf16 [M][K]; W[n][k] = table[idx[n][k]], idx packed 6 bits per weight
// (each row a little-endian bit stream, index k at bits [6k, 6k + 6)), table
// 64 bf16 values.  "Fast Accuracy-Preserving RNNT Beam Search on Apple
// Silicon", §1.3: the encoders store their weights as 64-entry lookup tables
// (6-bit palettes); the weight bytes fall from 2 to 0.75 per weight.
//
// One CTA per 128 x 64 output tile, 8 warps:
//   warp 0 lane 0  TMA producer: per 64-wide K slice, the A tile (128 x 64
//                  bf16, 128-byte swizzle) and the packed index tile (64 rows x
//                  48 bytes) into a 4-stage ring (barrier `full`);
//   warps 2-3      decoders: thread r turns weight row r's 48 bytes into 64
//                  table values and writes them in the 128-byte-swizzled
//                  K-major layout the tensor core reads (16-byte chunk c of row
//                  r at byte r * 128 + ((c ^ (r & 7)) * 16) of the 1024-aligned
//                  tile, the layout the TMA writes for the A tiles), then
//                  fences its shared-memory writes for the async proxy and
//                  arrives on `ready` (64 arrivals per stage);
//   warp 1 lane 0  MMA issuer: waits for `full` and `ready`, issues 4
//                  tcgen05.mma (K = 16 each), commits to `empty`;
//   all warps      epilogue: TMEM -> registers (+ bias) -> fp32 rows of C.
// Every wait is bounded; a wait that gives up latches CAC_E_TIMEOUT in the
// optional status word, and the CTA unwinds without storing any of its tile.
#include <cudaTypedefs.h>

#include <mutex>

#include "cac.h"
#include "cac_ops.h"
#include "gemm.cuh"

namespace cac {
namespace {

constexpr int PBM = 128, PBN = 64, PBK = 64, PST = 4, PTHREADS = 256;
constexpr int PA_TILE = PBM * PBK * 2;     // 16 KB
constexpr int PB_TILE = PBN * PBK * 2;     // 8 KB decoded
constexpr int PP_ROW = PBK * 6 / 8;        // 48 packed bytes per row and slice
constexpr int PP_TILE = PBN * PP_ROW;      // 3 KB packed
constexpr int PSMEM = PST * (PA_TILE + PB_TILE + PP_TILE) + 1024 /*align*/ + 512 /*barriers, table*/;

__global__ void __launch_bounds__(PTHREADS, 1)
    gemm_palette_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmP, int M,
                        int K, const uint16_t* table, const float* bias, float* C, int ldc, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + PST * PA_TILE;
    uint8_t* sP = sB + PST * PB_TILE;
    uint64_t* full = reinterpret_cast<uint64_t*>(sP + PST * PP_TILE);
    uint64_t* ready = full + PST;
    uint64_t* empty = ready + PST;
    uint64_t* accb = empty + PST;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
    uint16_t* tab = reinterpret_cast<uint16_t*>(tmem_slot + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * PBM, n0 = blockIdx.x * PBN;
    const int nk = K / PBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < PST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&ready[s], 64);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accb, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmP);
    }
    if (threadIdx.x < 64) tab[threadIdx.x] = table[threadIdx.x];
    if (warp == 1) tmem_alloc(tmem_slot, PBN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (warp == 0 && lane == 0) {
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % PST;
            const uint32_t ph = (kb / PST) & 1;
            if (kb >= PST && !mbar_wait(&empty[s], ph ^ 1)) { ok = false; break; }
            mbar_expect_tx(&full[s], PA_TILE + PP_TILE);
            tma_load_2d(sA + s * PA_TILE, &tmA, kb * PBK, m0, &full[s]);
            tma_load_2d(sP + s * PP_TILE, &tmP, kb * PP_ROW, n0, &full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        constexpr uint32_t idesc = idesc_bf16_f32(PBM, PBN);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % PST;
            const uint32_t ph = (kb / PST) & 1;
            if (!mbar_wait(&full[s], ph) || !mbar_wait(&ready[s], ph)) { ok = false; break; }
            tc_fence_after();
            const uint64_t ad = sdesc_k_sw128(sA + s * PA_TILE);
            const uint64_t bd = sdesc_k_sw128(sB + s * PB_TILE);
#pragma unroll
            for (int kk = 0; kk < PBK / 16; ++kk) tc_mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
            tc_commit(&empty[s]);
        }
        tc_commit(accb);
    } else if (warp == 2 || warp == 3) {
        const int r = threadIdx.x - 64;  // weight row of the tile
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % PST;
            const uint32_t ph = (kb / PST) & 1;
            if (!mbar_wait(&full[s], ph)) { ok = false; break; }
            const uint8_t* pk = sP + s * PP_TILE + r * PP_ROW;
            uint8_t* out = sB + s * PB_TILE + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // 8 indices = 6 bytes -> one 16-byte chunk of 8 bf16
                uint64_t v = 0;
#pragma unroll
                for (int q = 0; q < 6; ++q) v |= (uint64_t)pk[c * 6 + q] << (8 * q);
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = (uint32_t)tab[(v >> (12 * e)) & 63] | ((uint32_t)tab[(v >> (12 * e + 6)) & 63] << 16);
                *reinterpret_cast<uint4*>(out + ((c ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&ready[s]);
        }
    }
    __syncwarp();
    if (!mbar_wait(accb, 0)) ok = false;
    // a wait that gave up in any thread voids the whole tile: no thread stores
    const bool tile_ok = __syncthreads_or(!ok) == 0;
    tc_fence_after();
    const int quarter = warp & 3, half = warp >> 2;
    const int row = m0 + quarter * 32 + lane;
    {
        const int c = half * (PBN / 2);
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, v);
        if (tile_ok && row < M) {
            float* dst = C + (long long)row * ldc + n0 + c;
#pragma unroll
            for (int k = 0; k < 32; ++k) dst[k] = v[k] + (bias ? __ldg(bias + n0 + c + k) : 0.f);
        }
    }
    if (!ok) latch_error(status, CAC_E_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, PBN);
}

}  // namespace
}  // namespace cac

using namespace cac;

extern "C" int cac_op_gemm_palette(int M, int N, int K, const void* A, const void* packed, const void* table,
                                   const float* bias, float* C, int* status, void* stream) {
    if (M < 1 || N < PBN || K < PBK || N % PBN || K % PBK || !A || !packed || !table || !C) return CAC_E_INVAL;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(packed) | reinterpret_cast<uintptr_t>(C)) &
            15 ||
        (reinterpret_cast<uintptr_t>(table) & 1) || (reinterpret_cast<uintptr_t>(bias) & 3))
        return CAC_E_ALIGN;
    CUtensorMap ta, tp;
    if (!make_tmap_bf16(&ta, A, K, M, (uint64_t)K * 2, PBM) ||
        !make_tmap_packed(&tp, packed, (uint64_t)K * 3 / 4, (uint64_t)N))
        return CAC_E_CUDA;
    static bool attr = false;
    if (!attr) {
        if (cudaFuncSetAttribute(gemm_palette_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PSMEM) !=
            cudaSuccess)
            return CAC_E_CUDA;
        attr = true;
    }
    gemm_palette_kernel<<<dim3(N / PBN, (M + PBM - 1) / PBM), PTHREADS, PSMEM, static_cast<cudaStream_t>(stream)>>>(
        ta, tp, M, K, static_cast<const uint16_t*>(table), bias, C, N, status);
    return cudaGetLastError() == cudaSuccess ? CAC_OK : CAC_E_CUDA;
}
