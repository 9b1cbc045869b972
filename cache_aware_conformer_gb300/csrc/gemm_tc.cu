// tcgen05 / TMEM / TMA GEMM for sm_103a: C = A * B^T, bf16 operands, fp32
// accumulation in tensor memory, fused epilogue read back with tcgen05.ld.
//
// One CTA computes a 128 x BN output tile with 8 warps:
//   warp 0 lane 0  TMA producer: 64-wide K slices of A (128 rows) and B (BN rows)
//                  into a STAGES-deep ring of 128-byte-swizzled smem tiles;
//   warp 1 lane 0  MMA issuer: 4 x tcgen05.mma (K = 16 each) per slice, then
//                  tcgen05.commit to release the slice back to the producer;
//   warp 1         also owns the TMEM allocation (BN fp32 columns);
//   warps 0-7      epilogue: warp w reads TMEM lanes 32(w%4)..+31 (output rows),
//                  column half w/4, in 32-column chunks, and applies the fused
//                  epilogue.  Eight warps (two per scheduler) keep the
//                  epilogue's dependent arithmetic from stalling one warp per
//                  scheduler.  At BN = 64, eight stages put K = 512 in flight
//                  at once (one TMA round trip per tile); the epilogue warps
//                  load bias and residual rows while the main loop runs.
// Split operands: with SPLIT the A slice is a (hi, lo) pair of bf16 tiles and
// each slice issues 8 MMAs (hi then lo against the same B tile), so an fp32
// activation enters the product with ~16 significant bits while the
// contraction stays bf16 x bf16 with fp32 accumulation.
// Split-K: the `splits` CTAs of one output tile form a thread-block cluster
// along z, each accumulating a contiguous range of K slices.  Once every
// rank's main loop is done (a cluster barrier), ranks > 0 store their fp32
// partial tiles into rank 0's (now idle) pipeline shared memory over
// distributed shared memory; after a second barrier rank 0 adds them in rank
// order (deterministic) and runs the fused epilogue once.
// Every mbarrier wait is bounded; a wait that gives up latches
// CAC_E_TIMEOUT in the status word and the CTA unwinds without hanging.
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm.cuh"

namespace cac {

namespace {
constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_TILE = BM * BK * 2;  // bytes

// SPLIT: the A operand is a split pair (hi, lo) of bf16 tiles per K slice (hi
// at column k, lo at column K + k of the A tensor map); both are multiplied by
// the same B tile into the same accumulator.
// WIN (the fused GLU + depthwise-conv epilogue at BN = 64): a shared-memory copy
// of the conv-ring rows of the tile's streams, [stream][slot][32 channels]
// bf16 for up to 64 streams (two or more frames per stream), loaded by the
// idle warps before the wait on the previous kernel (the rows were written a
// step earlier); one ring stage fewer makes room for it.
// PAL (BN = 64): the weights are 6-bit palette indices (64 rows x 48 bytes per
// K slice, loaded by TMA) that warps 2-3 decode into the bf16 B tile through
// the 64-entry table of the tile's rows.
template <int BN, int SPLIT, int KIND, int PAL = 0>
struct TcCfg {
    static_assert(!PAL || BN == 64, "palette tiles are 64 rows");
    static constexpr bool HAS_WIN = KIND == EPI_GLUDW && BN == 64;
    static constexpr int P_TILE = PAL ? 64 * 48 : 0;
    static constexpr int WIN = HAS_WIN ? 64 * 8 * 32 * 2 : 0;
    static constexpr int PRM = HAS_WIN ? (12 * 32 + 64) * 4 : 0;  // conv constants and LayerNorm column sums
    static constexpr int B_TILE = BN * BK * 2;
    static constexpr int A_TILES = A_TILE * (1 + SPLIT);
    static constexpr int STAGE = A_TILES + B_TILE + P_TILE;
    static constexpr int TX = A_TILES + (PAL ? P_TILE : B_TILE);  // bytes the TMA brings per stage
    static constexpr int STAGES = SPLIT ? ((BN == 256) ? 3 : (BN == 128 ? 4 : (HAS_WIN ? 4 : 5)))
                                        : ((BN == 256) ? 4 : (BN == 128 ? 6 : 8));
    static constexpr int SMEM = STAGES * STAGE + 1024 /*align slack*/ + 256 /*barriers*/ + BM * 8 /*row stats*/ + WIN + PRM +
                                (PAL ? 128 : 0) /*table*/;
    static_assert(BN != 64 || STAGES * A_TILES >= 3 * BN * BM * 4, "split-K partial tiles must fit the A ring");
    static_assert(BN != 128 || STAGES * A_TILES >= 3 * 32 * BM * 4, "owner-mode partial chunks must fit the A ring");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};
}  // namespace

constexpr int TC_THREADS = 256;

template <int BN, int KIND, class TAct, int SPLIT, int PAL>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M, int N,
                   int K, int conv_C, EpiParams ep, const uint16_t* pal_tab, int* status) {
    using C = TcCfg<BN, SPLIT, KIND, PAL>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + C::STAGES * C::A_TILES;
    uint8_t* sP = sB + C::STAGES * C::B_TILE;  // PAL: packed index tiles
    uint64_t* full = reinterpret_cast<uint64_t*>(sP + C::STAGES * C::P_TILE);
    uint64_t* empty = full + C::STAGES;
    uint64_t* accb = empty + C::STAGES;
    uint64_t* ready = accb + 2;  // PAL: [STAGES] decoded B tiles (64 arrivals)
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
    // LayerNorm statistics of the tile's rows, computed once per row by warps
    // 2-5 while the main loop runs (warps 0 and 1 are busy in it)
    float2* rowstat = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(full) + 256);
    bf16* win = reinterpret_cast<bf16*>(rowstat + BM);  // C::WIN bytes
    float* prm = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(win) + C::WIN);  // C::PRM bytes
    uint16_t* ptab = reinterpret_cast<uint16_t*>(reinterpret_cast<uint8_t*>(prm) + C::PRM);  // PAL: 64 entries
    // warps free during the main loop: 2-7, or 4-7 when 2-3 decode palette tiles
    constexpr int FREE0 = PAL ? 4 : 2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    const int splits = gridDim.z;
    const uint32_t crank = splits > 1 ? cluster_rank() : 0;
    const int nk_all = K / BK;
    const int kb0 = (int)(crank * nk_all / splits), kb1 = (int)((crank + 1) * nk_all / splits);
    const int nk = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accb, 1);
        if (PAL)
            for (int s = 0; s < C::STAGES; ++s) mbar_init(&ready[s], 64);
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (PAL && threadIdx.x < 64) ptab[threadIdx.x] = pal_tab[(size_t)(n0 / 64) * 64 + threadIdx.x];
    if (warp == 1) tmem_alloc(tmem_slot, BN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    bool ok = true;
    if (warp == 0 && lane == 0) {
        // weights never depend on the previous kernel: start the first stages' B
        // tiles before waiting for it, then the activations
        const int pre = nk < C::STAGES ? nk : C::STAGES;
        for (int kb = 0; kb < pre; ++kb) {
            mbar_expect_tx(&full[kb], C::TX);
            if (PAL) tma_load_2d(sP + kb * C::P_TILE, &tmB, (kb0 + kb) * 48, n0, &full[kb]);
            else tma_load_2d(sB + kb * C::B_TILE, &tmB, (kb0 + kb) * BK, n0, &full[kb]);
        }
        pdl_wait();
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % C::STAGES;
            const uint32_t ph = (kb / C::STAGES) & 1;
            const int k0 = (kb0 + kb) * BK;
            if (kb >= pre) {
                if (!mbar_wait(&empty[s], ph ^ 1)) { ok = false; break; }
                mbar_expect_tx(&full[s], C::TX);
                if (PAL) tma_load_2d(sP + s * C::P_TILE, &tmB, (kb0 + kb) * 48, n0, &full[s]);
                else tma_load_2d(sB + s * C::B_TILE, &tmB, k0, n0, &full[s]);
            }
            if (conv_C) {
                const int tap = k0 / conv_C;
                tma_load_3d(sA + s * C::A_TILES, &tmA, k0 - tap * conv_C, tap & 1, m0 + (tap >> 1), &full[s]);
                if (SPLIT)
                    tma_load_3d(sA + s * C::A_TILES + A_TILE, &tmA, conv_C + k0 - tap * conv_C, tap & 1,
                                m0 + (tap >> 1), &full[s]);
            } else {
                tma_load_2d(sA + s * C::A_TILES, &tmA, k0, m0, &full[s]);
                if (SPLIT) tma_load_2d(sA + s * C::A_TILES + A_TILE, &tmA, K + k0, m0, &full[s]);
            }
        }
    } else if (warp == 1 && lane == 0) {
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % C::STAGES;
            const uint32_t ph = (kb / C::STAGES) & 1;
            if (!mbar_wait(&full[s], ph) || (PAL && !mbar_wait(&ready[s], ph))) { ok = false; break; }
            tc_fence_after();
            const uint64_t ad = sdesc_k_sw128(sA + s * C::A_TILES);
            const uint64_t bd = sdesc_k_sw128(sB + s * C::B_TILE);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                // +32 bytes along K inside the swizzle atom = +2 in the encoded start address
                tc_mma_bf16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
            }
            if (SPLIT) {
                const uint64_t al = sdesc_k_sw128(sA + s * C::A_TILES + A_TILE);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) tc_mma_bf16(tmem, al + 2 * kk, bd + 2 * kk, idesc, 1u);
            }
            tc_commit(&empty[s]);
        }
        tc_commit(accb);
    } else if (PAL && (warp == 2 || warp == 3)) {
        // decoders: thread r turns weight row r's 48 packed bytes of each K slice
        // (index k at bits [6k, 6k + 6)) into 64 table values, written in the
        // 128-byte-swizzled K-major layout the tensor core reads (16-byte chunk c
        // of row r at byte r * 128 + ((c ^ (r & 7)) << 4), as the TMA writes the
        // A tiles)
        const int r = threadIdx.x - 64;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % C::STAGES;
            const uint32_t ph = (kb / C::STAGES) & 1;
            if (!mbar_wait(&full[s], ph)) { ok = false; break; }
            // the row's 48 bytes as three 16-byte loads (rows 48 bytes apart, the
            // tile 1024-aligned), then 6 bytes = 8 indices per 16-byte output chunk
            const uint4* pk4 = reinterpret_cast<const uint4*>(sP + s * C::P_TILE + r * 48);
            uint32_t wd[12];
#pragma unroll
            for (int q = 0; q < 3; ++q) {
                const uint4 t = pk4[q];
                wd[4 * q] = t.x; wd[4 * q + 1] = t.y; wd[4 * q + 2] = t.z; wd[4 * q + 3] = t.w;
            }
            uint8_t* out = sB + s * C::B_TILE + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // 8 indices = 6 bytes -> one 16-byte chunk of 8 bf16
                // bytes 6c .. 6c + 5 of the row, little-endian
                const int b0 = 6 * c, w0 = b0 >> 2, sh = 8 * (b0 & 3);
                const uint64_t lo = (uint64_t)wd[w0] | ((uint64_t)wd[w0 + 1] << 32);
                const uint64_t hi = w0 + 2 < 12 ? (uint64_t)wd[w0 + 2] : 0ull;
                const uint64_t v = ((lo >> sh) | (sh ? hi << (64 - sh) : 0ull)) & 0xFFFFFFFFFFFFull;
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = (uint32_t)ptab[(v >> (12 * e)) & 63] | ((uint32_t)ptab[(v >> (12 * e + 6)) & 63] << 16);
                *reinterpret_cast<uint4*>(out + ((c ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&ready[s]);
        }
    }
    // conv-ring window of the tile's streams (GLU + depthwise epilogue): the
    // slots hold frames of earlier steps, final before this kernel started, so
    // the idle warps copy them while the previous kernel finishes, with the
    // per-channel constants of the tile's 32 channels and the LayerNorm
    // column sums of its 64 columns
    const bool use_win = C::HAS_WIN && ep.nq >= 2;
    if constexpr (C::HAS_WIN) {
        if (warp >= FREE0) {
            const int C0 = n0 >> 1;
            for (int i = threadIdx.x - 32 * FREE0; i < 12 * 32 + 64; i += TC_THREADS - 32 * FREE0) {
                float v;
                if (i < 9 * 32) v = __ldg(ep.dw_wT + (long long)(i >> 5) * ep.D + C0 + (i & 31));
                else if (i < 10 * 32) v = __ldg(ep.dw_bias + C0 + i - 9 * 32);
                else if (i < 11 * 32) v = __ldg(ep.dw_gamma + C0 + i - 10 * 32);
                else if (i < 12 * 32) v = __ldg(ep.dw_beta + C0 + i - 11 * 32);
                else v = ep.ln_colsum ? __ldg(ep.ln_colsum + n0 + i - 12 * 32) : 0.f;
                prm[i] = v;
            }
        }
        if (use_win && warp >= FREE0) {
            // 16-byte pieces idx = (stream, slot, quarter of 8 channels), in batches
            // whose stream ids and then ring rows are all requested before any
            // is used (one dependent round trip each per batch)
            constexpr int LT = TC_THREADS - 32 * FREE0, PER = PAL ? 8 : 6;
            const int nS = BM / ep.nq, sb0 = m0 / ep.nq, C0 = n0 >> 1, t = threadIdx.x - 32 * FREE0;
            const bf16* ring = static_cast<const bf16*>(ep.dw_ring);
            uint4* w4 = reinterpret_cast<uint4*>(win);
            for (int j0 = 0; j0 * LT < nS * 32; j0 += PER) {
                int id[PER];
#pragma unroll
                for (int j = 0; j < PER; ++j) {
                    const int idx = t + (j0 + j) * LT, b = sb0 + (idx >> 5);
                    id[j] = (idx < nS * 32 && b * ep.nq < ep.dw_rows) ? ep.ids[b] : -1;
                }
                uint4 v[PER];
#pragma unroll
                for (int j = 0; j < PER; ++j) {
                    const int idx = t + (j0 + j) * LT, slot = (idx >> 2) & 7, q = idx & 3;
                    v[j] = make_uint4(0u, 0u, 0u, 0u);
                    if (id[j] >= 0 && id[j] < ep.n_streams)  // an id out of range is latched by epi_prefetch
                        v[j] = *reinterpret_cast<const uint4*>(ring + (long long)id[j] * ep.dw_sstride +
                                                               (long long)slot * ep.D + C0 + 8 * q);
                }
#pragma unroll
                for (int j = 0; j < PER; ++j) {
                    const int idx = t + (j0 + j) * LT;
                    if (idx < nS * 32) w4[idx] = v[j];
                }
            }
        }
    }
    __syncwarp();
    pdl_wait();  // the epilogue reads/writes buffers of earlier kernels
    const int quarter = warp & 3, half = warp >> 2;
    const int rloc = quarter * 32 + lane;
    const int row = m0 + rloc;
    // owner mode (BN = 128, 4-way split-K): rank r reduces and finishes the
    // tile's 32-column chunk r; otherwise rank 0 finishes the whole tile
    const bool owner = BN == 128 && splits == 4;
    const bool finisher = owner ? half == 0 : crank == 0;
    const int c_first = owner ? 32 * (int)crank : half * (BN / 2);
    EpiPre pre;
    const bool row_stats = ep.ln_stats != nullptr && (owner || crank == 0);
    if (finisher && (row < M || KIND == EPI_GLUDW)) epi_prefetch<KIND>(ep, row, n0 + c_first, pre, !row_stats);
    if (row_stats && warp >= FREE0 && warp < FREE0 + 4)
        rowstat[(warp - FREE0) * 32 + lane] = epi_row_stats(ep, m0 + (warp - FREE0) * 32 + lane);

    if (!mbar_wait(accb, 0)) ok = false;
    if constexpr (C::HAS_WIN) {
        if (!row_stats) __syncthreads();  // the conv-ring window and constants are in shared memory
    }
    if (row_stats) {
        __syncthreads();  // the row statistics are in shared memory
        if (row < M || KIND == EPI_GLUDW) epi_apply_stats(rowstat[rloc], pre);
    }
    pdl_trigger();  // main loop done: let the next kernel launch while the epilogue runs
    tc_fence_after();
    // split-K: the partial tiles of ranks 1 .. splits-1, [rank - 1][BN columns][128
    // rows] fp32, land in rank 0's pipeline buffers (idle once every rank's main
    // loop is done)
    float* part = reinterpret_cast<float*>(sA);
    static_assert(KIND == EPI_GLUDW || C::STAGES * C::B_TILE >= 8 * EPI_STAGE_FLOATS * 4, "epilogue staging");
    float* stage = reinterpret_cast<float*>(sB) + warp * EPI_STAGE_FLOATS;
    if (splits > 1) {
        cluster_sync();  // every rank's main loop is done: the finishers' rings take the partials
        if (owner) {
            // this rank's partial of chunk q goes to rank q, into slot (its rank
            // among q's three peers); half 0 pushes the first and third other
            // chunk, half 1 the second
#pragma unroll 1
            for (int i = half; i < 3; i += 2) {
                const int q = i + (i >= (int)crank ? 1 : 0);
                const int slot = (int)crank < q ? (int)crank : (int)crank - 1;
                const uint32_t dst = dsmem_addr(part + (size_t)slot * 32 * BM + rloc, (uint32_t)q);
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(32 * q), v);
#pragma unroll
                for (int k = 0; k < 32; ++k) st_dsmem_f32(dst + (uint32_t)(k * BM) * 4u, v[k]);
            }
        } else if (crank != 0) {
            // pushed with remote stores (a warp writes one 128-byte column
            // segment per store), so that rank 0 adds them from its own memory
            const uint32_t dst = dsmem_addr(part + (size_t)(crank - 1) * BN * BM + rloc, 0);
#pragma unroll 1
            for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
                float v[32];
                tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, v);
#pragma unroll
                for (int k = 0; k < 32; ++k) st_dsmem_f32(dst + (uint32_t)((c + k) * BM) * 4u, v[k]);
            }
        }
        cluster_sync();  // the partials are in the finishers' shared memory
    }
    if (owner) {
        if (half == 0) {
            // the chunk's four partials added in rank order (the same order as
            // rank 0 finishing the whole tile: bit-identical results)
            float own[32], v[32];
            tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c_first, own);
#pragma unroll 1
            for (int rr = 0; rr < 4; ++rr) {
                const float* pr = part + (size_t)(rr < (int)crank ? rr : rr - 1) * 32 * BM + rloc;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float t = rr == (int)crank ? own[k] : pr[k * BM];
                    v[k] = rr == 0 ? t : v[k] + t;
                }
            }
            const bool live = ok && row < M;
            if constexpr (KIND != EPI_GLUDW) epilogue32<KIND, TAct>(ep, row, n0 + c_first, v, pre, stage, live);
        }
    } else if (crank == 0) {
#pragma unroll 1
        for (int c = half * (BN / 2); c < (half + 1) * (BN / 2); c += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c, v);
            for (int rr = 1; rr < splits; ++rr) {  // in rank order (deterministic)
                const float* pr = part + (size_t)(rr - 1) * BN * BM + rloc;
#pragma unroll
                for (int k = 0; k < 32; ++k) v[k] += pr[(c + k) * BM];
            }
            if constexpr (KIND == EPI_GLUDW) {
                if (c != c_first) {  // bias only: any row
                    epi_prefetch<KIND>(ep, row, n0 + c, pre, !row_stats);
                    if (row_stats) epi_apply_stats(rowstat[rloc], pre);
                }
                epilogue_gludw(ep, row, ok && row < M, n0 + c, v, pre,
                               use_win ? win + (rloc / ep.nq) * 256 + (c >> 1) : nullptr,
                               C::HAS_WIN ? prm + (c >> 1) : nullptr, C::HAS_WIN ? prm + 12 * 32 + c : nullptr);
            } else {
                // every lane: the row stores go through this warp's slice of the
                // (idle) B ring
                const bool live = ok && row < M;
                if (c != c_first && live) {
                    epi_prefetch<KIND>(ep, row, n0 + c, pre, !row_stats);
                    if (row_stats) epi_apply_stats(rowstat[rloc], pre);
                }
                epilogue32<KIND, TAct>(ep, row, n0 + c, v, pre, stage, live);
            }
        }
    }
    if (!ok) latch_error(status, CAC_E_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, BN);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

bool make_tmap_bf16_conv(CUtensorMap* tm, const void* base, uint64_t C, uint64_t pairs, uint32_t box_rows) {
    std::call_once(g_encode_once, load_encode);
    if (!g_encode) return false;
    if ((reinterpret_cast<uintptr_t>(base) & 15) || (C % 64) || pairs == 0) return false;
    cuuint64_t dims[3] = {C, 2, pairs};
    cuuint64_t strides[2] = {C * 2, C * 4};
    cuuint32_t box[3] = {64, 1, box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_bf16_blocks(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t blocks,
                           uint64_t block_stride_bytes, uint32_t box_rows) {
    std::call_once(g_encode_once, load_encode);
    if (!g_encode) return false;
    if ((reinterpret_cast<uintptr_t>(base) & 15) || (block_stride_bytes & 15) || rows == 0 || blocks == 0 ||
        box_rows == 0 || box_rows > 256 || box_rows > rows)
        return false;
    cuuint64_t dims[3] = {64, rows, blocks};
    cuuint64_t strides[2] = {128, block_stride_bytes};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
                    uint32_t box_rows) {
    std::call_once(g_encode_once, load_encode);
    if (!g_encode) return false;
    if ((reinterpret_cast<uintptr_t>(base) & 15) || (row_stride_bytes & 15) || rows == 0 || inner < 64) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, int KIND, int SPLIT, int PAL>
static cudaError_t launch_bn_kind(const CUtensorMap* tmA, const CUtensorMap* tmB, int M, int N, int K, int conv_C,
                                  int splits, const EpiParams& ep, const uint16_t* pal_tab, int* status,
                                  cudaStream_t s) {
    using C = TcCfg<BN, SPLIT, KIND, PAL>;
    auto kern = gemm_tc_kernel<BN, KIND, bf16, SPLIT, PAL>;
    static bool attr_set = false;  // per instantiation, per process
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    return launch_k(kern, dim3(N / BN, (M + BM - 1) / BM, splits), dim3(TC_THREADS), C::SMEM, s, splits, *tmA, *tmB,
                    M, N, K, conv_C, ep, pal_tab, status);
}

template <int BN, int PAL>
static cudaError_t launch_bn(const CUtensorMap* tmA, const CUtensorMap* tmB, int M, int N, int K, int cc, int sp,
                             int a_split, const EpiParams& ep, const uint16_t* pt, int* status, cudaStream_t s) {
    if (a_split) {
        // split operands: LayerNorm outputs, the attention output, the subsampling windows
        switch (ep.kind) {
            case EPI_STORE: return launch_bn_kind<BN, EPI_STORE, 1, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
            case EPI_RESID: return launch_bn_kind<BN, EPI_RESID, 1, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
            case EPI_GLU: return launch_bn_kind<BN, EPI_GLU, 1, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
            case EPI_QKV: return launch_bn_kind<BN, EPI_QKV, 1, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
            case EPI_SUB: return launch_bn_kind<BN, EPI_SUB, 1, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
            case EPI_GLUDW: return launch_bn_kind<BN, EPI_GLUDW, 1, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (ep.kind) {
        case EPI_STORE: return launch_bn_kind<BN, EPI_STORE, 0, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
        case EPI_RESID: return launch_bn_kind<BN, EPI_RESID, 0, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
        case EPI_GLU: return launch_bn_kind<BN, EPI_GLU, 0, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
        case EPI_QKV: return launch_bn_kind<BN, EPI_QKV, 0, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
        case EPI_SUB: return launch_bn_kind<BN, EPI_SUB, 0, PAL>(tmA, tmB, M, N, K, cc, sp, ep, pt, status, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc(const CUtensorMap* tmA, const CUtensorMap* tmB, int M, int N, int K, int BN, int conv_C,
                           int splits, int a_split, const EpiParams& ep, int* status, cudaStream_t s,
                           const uint16_t* pal_tab) {
    if (M <= 0) return cudaSuccess;
    if (K % BK || K <= 0 || N % BN || !ep.act_bf16) return cudaErrorInvalidValue;
    if (conv_C && (conv_C % BK || K != 3 * conv_C)) return cudaErrorInvalidValue;
    if (splits < 1 || splits > 4 || splits > K / BK) return cudaErrorInvalidValue;
    // rank 0's ring holds three 128 x 64 partials; at BN = 128 the four ranks
    // each finish a 32-column chunk (owner mode)
    if (splits > 1 && !(BN == 64 || (BN == 128 && splits == 4))) return cudaErrorInvalidValue;
    if (ep.kind == EPI_GLUDW && (splits != 1 || !a_split || ep.nq < 1 || 32 % ep.nq || 2 * ep.D != N || ep.D % 16))
        return cudaErrorInvalidValue;
    if (pal_tab) {  // palette weights: 64-row tiles, tmB over the packed indices
        if (BN != 64) return cudaErrorInvalidValue;
        return launch_bn<64, 1>(tmA, tmB, M, N, K, conv_C, splits, a_split, ep, pal_tab, status, s);
    }
    switch (BN) {
        case 64: return launch_bn<64, 0>(tmA, tmB, M, N, K, conv_C, splits, a_split, ep, nullptr, status, s);
        case 128: return launch_bn<128, 0>(tmA, tmB, M, N, K, conv_C, splits, a_split, ep, nullptr, status, s);
        case 256: return launch_bn<256, 0>(tmA, tmB, M, N, K, conv_C, splits, a_split, ep, nullptr, status, s);
    }
    return cudaErrorInvalidValue;
}

// packed 6-bit indices [rows][row_bytes] (row_bytes = 3K/4), box of 48 bytes x 64 rows, no swizzle
bool make_tmap_packed(CUtensorMap* tm, const void* base, uint64_t row_bytes, uint64_t rows) {
    std::call_once(g_encode_once, load_encode);
    if (!g_encode) return false;
    if ((reinterpret_cast<uintptr_t>(base) & 15) || (row_bytes % 16) || rows == 0) return false;
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {48, 64};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace cac
