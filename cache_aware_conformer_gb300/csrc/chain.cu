// Persistent chain kernel: the projections and LayerNorms of the streaming step
// between two attention launches ("True streaming encode — implementation
// spec", §Per-chunk flow steps 2-4: FF1, ln -> Q/K/V, out-projection, pw1 +
// GLU + depthwise conv, pw2, FF2, ln_out, the joint projection) as one
// cooperative launch instead of one launch per projection.
//
// Work: phase p (chain.cuh) of row block r (128 rows) is split into tasks —
// 128 x 64 output tiles, each possibly one of `splits` K ranges, or 32-row
// LayerNorm groups.  Tasks are numbered phase by phase (row block, tile, split
// within a phase); CTA c takes tasks c, c + G, c + 2G, ... in that order.  A
// task of phase p > 0 waits (bounded) until phase p - 1 of its row block is
// complete (a counter per phase and row block, incremented once per finished
// tile or LayerNorm group).  Tasks only wait on earlier phases, every CTA is
// resident (cooperative launch) and takes its tasks in order, so every wait
// ends.
//
// Roles in each CTA (10 warps):
//   warp 0 lane 0  TMA producer: one continuous 4-stage ring over the CTA's
//                  tiles; a stage holds a 64-wide K slice of A (a split (hi,
//                  lo) pair when the phase's A is split) and of B.  The weight
//                  slices of a task's first stages are requested before its
//                  dependency wait; the activations after it.
//   warp 1 lane 0  MMA issuer: tcgen05.mma into one of two TMEM accumulators
//                  (128 x 64 fp32 each), so the epilogue of one tile overlaps
//                  the main loop of the next.
//   warps 2-9      epilogue: TMEM -> registers, split-K partials through the
//                  workspace (the last split to finish adds them in split
//                  order, then runs the epilogue: deterministic), the fused
//                  epilogue of gemm.cuh, completion count; LayerNorm tasks.
// Data written by one CTA and read by another inside the launch is read
// through L2 (__ldcg, or TMA after a proxy fence), after an acquire of the
// completion counter that the writer released.
// Every wait is bounded (about a second); a wait that gives up latches
// CAC_E_TIMEOUT and raises the abort word, and the CTAs unwind.
#include "chain.cuh"

namespace cac {

namespace {
constexpr int CBM = 128, CBN = 64, CBK = 64;
constexpr int C_ST = 4;
constexpr int C_A_TILE = CBM * CBK * 2;               // 16 KB
constexpr int C_B_TILE = CBN * CBK * 2;               // 8 KB
constexpr int C_STAGE = 2 * C_A_TILE + C_B_TILE;      // A hi | A lo | B
constexpr int C_EPI_WARPS = 8;
constexpr int C_THREADS = 32 * (2 + C_EPI_WARPS);
constexpr int C_OFF_STAGING = C_ST * C_STAGE;
constexpr int C_OFF_BAR = C_OFF_STAGING + C_EPI_WARPS * EPI_STAGE_FLOATS * 4;
constexpr int C_OFF_PH = C_OFF_BAR + 256;             // the phase table, copied once
constexpr int C_PH_BYTES = ((int)sizeof(ChainPhase) * CH_MAX_PHASES + 127) / 128 * 128;
constexpr int C_SMEM = C_OFF_PH + C_PH_BYTES + 1024 /*alignment slack*/;
static_assert(C_SMEM <= 227 * 1024, "shared memory");
static_assert(sizeof(ChainPhase) % 16 == 0, "phase table copied in 16-byte pieces");
constexpr long long SPIN_LIMIT = 1ll << 31;           // clock cycles (~1 s)

__device__ __forceinline__ int ld_acquire_i32(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int ld_relaxed_i32(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// bounded wait until *p >= target; false on timeout (latched) or abort.  Polls
// with relaxed loads (an acquire load per poll would keep invalidating the SM's
// L1) and acquires once the count is reached.
__device__ bool wait_count(const int* p, int target, const ChainCtl& c) {
    if (ld_acquire_i32(p) >= target) return true;
    const long long t0 = clock64();
    for (unsigned it = 0;; ++it) {
        if (ld_relaxed_i32(p) >= target) return ld_acquire_i32(p) >= target;
        __nanosleep(64);
        if ((it & 15u) == 15u) {
            if (*(volatile int*)c.abort) return false;
            if (clock64() - t0 > SPIN_LIMIT) {
                latch_error(c.status, CAC_E_TIMEOUT);
                atomicExch(c.abort, 1);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void fail(const ChainCtl& c) {
    latch_error(c.status, CAC_E_TIMEOUT);
    atomicExch(c.abort, 1);
}

// named barrier of the epilogue warps only
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(32 * C_EPI_WARPS) : "memory"); }
// the same barrier, returning whether v holds in every epilogue thread (so that
// all epilogue warps take the same branch after a bounded wait)
__device__ __forceinline__ bool epi_all(bool v) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.s32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\t"
        "selp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((int)v), "n"(32 * C_EPI_WARPS)
        : "memory");
    return r != 0;
}

// the task sequence of one role: phases in order, C_THREADS-independent
struct TaskSeq {
    int p = 0, start = 0, end = 0;
    __device__ void init(const ChainPhase* ph, int n_rb) { end = n_rb * ph[0].tasks_rb; }
    // moves to the phase holding global task g (g never decreases); false past the end
    __device__ bool seek(int g, const ChainPhase* ph, int n_ph, int n_rb) {
        while (g >= end) {
            if (++p >= n_ph) return false;
            start = end;
            end += n_rb * ph[p].tasks_rb;
        }
        return true;
    }
};

// ---------------------------------------------------------------------------
// LayerNorm rows (vectorized layout: lane holds columns 128 j + 4 lane + e)
// ---------------------------------------------------------------------------
template <int VPL>
__device__ __forceinline__ void ln_vals(float (&v)[VPL], int D, const float* g, const float* b) {
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) s += v[k];
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s / D;
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < VPL; ++k) {
        const float d = v[k] - mean;
        q += d * d;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float rstd = rsqrtf(q / D + 1e-5f);
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < VPL / 4; ++j) {
        const int c = 128 * j + 4 * lane;
        const float4 gg = __ldg(reinterpret_cast<const float4*>(g + c));
        const float4 bb = __ldg(reinterpret_cast<const float4*>(b + c));
        v[4 * j] = (v[4 * j] - mean) * rstd * gg.x + bb.x;
        v[4 * j + 1] = (v[4 * j + 1] - mean) * rstd * gg.y + bb.y;
        v[4 * j + 2] = (v[4 * j + 2] - mean) * rstd * gg.z + bb.z;
        v[4 * j + 3] = (v[4 * j + 3] - mean) * rstd * gg.w + bb.w;
    }
}

__device__ __forceinline__ uint2 pack4(float a, float b, float c, float d) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

template <int VPL>
__device__ __forceinline__ void store_act4(bf16* dst, long long row, int D, const float (&v)[VPL], int split) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < VPL / 4; ++j) {
        const int c = 128 * j + 4 * lane;
        const float a0 = v[4 * j], a1 = v[4 * j + 1], a2 = v[4 * j + 2], a3 = v[4 * j + 3];
        const uint2 h = pack4(a0, a1, a2, a3);
        if (split) {
            bf16* d = dst + row * 2 * D + c;
            *reinterpret_cast<uint2*>(d) = h;
            const __nv_bfloat162* hp = reinterpret_cast<const __nv_bfloat162*>(&h);
            const float2 f0 = __bfloat1622float2(hp[0]), f1 = __bfloat1622float2(hp[1]);
            *reinterpret_cast<uint2*>(d + D) = pack4(a0 - f0.x, a1 - f0.y, a2 - f1.x, a3 - f1.y);
        } else {
            *reinterpret_cast<uint2*>(dst + row * D + c) = h;
        }
    }
}

template <int VPL>
__device__ void ln_row_task(const ChainPhase& P, int row) {
    const int lane = threadIdx.x & 31, D = P.D;
    float v[VPL];
#pragma unroll
    for (int j = 0; j < VPL / 4; ++j) {
        const float4 t = __ldcg(reinterpret_cast<const float4*>(P.x + (long long)row * D + 128 * j + 4 * lane));
        v[4 * j] = t.x; v[4 * j + 1] = t.y; v[4 * j + 2] = t.z; v[4 * j + 3] = t.w;
    }
    ln_vals<VPL>(v, D, P.g1, P.b1);
    if (P.y_f32) {
        const long long orow = (long long)(row / P.grp) * P.grp_stride + (row % P.grp) + P.row_off;
#pragma unroll
        for (int j = 0; j < VPL / 4; ++j)
            *reinterpret_cast<float4*>(P.y_f32 + orow * D + 128 * j + 4 * lane) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    if (P.y_act) store_act4<VPL>(P.y_act, row, D, v, P.split);
    if (P.g2) {
        ln_vals<VPL>(v, D, P.g2, P.b2);
        store_act4<VPL>(P.z_act, row, D, v, P.split);
    }
}

// GEMM epilogue of one 32-column segment of one row, by kind
__device__ __forceinline__ void run_epilogue(const EpiParams& ep, int row, int M, int col, float (&v)[32],
                                             float* stage) {
    const bool live = row < M;
    EpiPre pre;
    switch (ep.kind) {
        case EPI_STORE:
            if (live) epi_prefetch<EPI_STORE>(ep, row, col, pre);
            epilogue32<EPI_STORE, bf16>(ep, row, col, v, pre, stage, live);
            break;
        case EPI_RESID:
            if (live) epi_prefetch<EPI_RESID>(ep, row, col, pre);
            epilogue32<EPI_RESID, bf16>(ep, row, col, v, pre, stage, live);
            break;
        case EPI_QKV:
            if (live) epi_prefetch<EPI_QKV>(ep, row, col, pre);
            epilogue32<EPI_QKV, bf16>(ep, row, col, v, pre, stage, live);
            break;
        case EPI_GLUDW:
            epi_prefetch<EPI_GLUDW>(ep, row, col, pre);
            epilogue_gludw(ep, row, live, col, v, pre, nullptr, nullptr, nullptr);
            break;
        default: break;
    }
}
}  // namespace

__global__ void __launch_bounds__(C_THREADS, 1)
    chain_kernel(const ChainPhase* __restrict__ gph, int n_ph, int M, ChainCtl c) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // the phase table lives in shared memory for the whole launch; only the TMA
    // copies use the tensor maps of the global copy (gph)
    ChainPhase* ph = reinterpret_cast<ChainPhase*>(smem + C_OFF_PH);
    {
        const int4* src = reinterpret_cast<const int4*>(gph);
        int4* dst = reinterpret_cast<int4*>(ph);
        const int n16 = n_ph * (int)sizeof(ChainPhase) / 16;
        for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = __ldg(src + i);
    }
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C_OFF_BAR);
    uint64_t* empty = full + C_ST;
    uint64_t* tfull = empty + C_ST;   // [2] accumulator ready for the epilogue
    uint64_t* tempty = tfull + 2;     // [2] accumulator drained by the epilogue
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
    int* last_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_rb = (M + CBM - 1) / CBM;
    const int G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C_ST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], C_EPI_WARPS);
        }
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, 2 * CBN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            TaskSeq ts;
            ts.init(ph, n_rb);
            int it = 0;  // K slices issued so far (ring position)
            bool ok = true;
            for (int g = blockIdx.x; ok && ts.seek(g, ph, n_ph, n_rb); g += G) {
                const ChainPhase& P = ph[ts.p];
                const ChainPhase& G = gph[ts.p];  // tensor maps: global memory
                const int local = g - ts.start, rb = local / P.tasks_rb, r = local - rb * P.tasks_rb;
                if (P.op != CH_GEMM) continue;
                const int tile = r / P.splits, sp = r - tile * P.splits;
                const int m0 = rb * CBM, n0 = tile * CBN;
                const int nk_all = P.K / CBK;
                const int kb0 = sp * nk_all / P.splits, kb1 = (sp + 1) * nk_all / P.splits, nk = kb1 - kb0;
                const uint32_t bytes = C_A_TILE * (1 + P.a_split) + C_B_TILE;
                const int pre = nk < C_ST ? nk : C_ST;
                // weights first: they never depend on an earlier phase.  Their
                // bytes may land before the stage is armed (the transaction count
                // goes negative; the phase cannot complete before the arrival).
                for (int j = 0; j < pre && ok; ++j) {
                    const int s = (it + j) % C_ST;
                    if (it + j >= C_ST && !mbar_wait(&empty[s], (((it + j) / C_ST) & 1) ^ 1)) { ok = false; break; }
                    tma_load_2d(smem + s * C_STAGE + 2 * C_A_TILE, &G.tb, (kb0 + j) * CBK, n0, &full[s]);
                }
                if (!ok) break;
                if (ts.p > 0 && !wait_count(c.cnt + (ts.p - 1) * CH_MAX_RB + rb, ph[ts.p - 1].done_rb, c)) {
                    ok = false;
                    break;
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");  // the writers' generic stores, for TMA
                // every stage is armed (a release) after the acquire above, so the
                // MMA issuer and, through it, the epilogue are ordered after it
                for (int j = 0; j < nk; ++j) {
                    const int s = (it + j) % C_ST;
                    uint8_t* st = smem + s * C_STAGE;
                    const int k0 = (kb0 + j) * CBK;
                    if (j >= pre) {
                        if (!mbar_wait(&empty[s], (((it + j) / C_ST) & 1) ^ 1)) { ok = false; break; }
                        tma_load_2d(st + 2 * C_A_TILE, &G.tb, k0, n0, &full[s]);
                    }
                    mbar_expect_tx(&full[s], bytes);
                    tma_load_2d(st, &G.ta, k0, m0, &full[s]);
                    if (P.a_split) tma_load_2d(st + C_A_TILE, &G.ta, P.K + k0, m0, &full[s]);
                }
                it += nk;
            }
            if (!ok) fail(c);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(CBM, CBN);
            TaskSeq ts;
            ts.init(ph, n_rb);
            int it = 0, lt = 0;
            bool ok = true;
            for (int g = blockIdx.x; ok && ts.seek(g, ph, n_ph, n_rb); g += G) {
                const ChainPhase& P = ph[ts.p];
                if (P.op != CH_GEMM) continue;
                const int local = g - ts.start, rb = local / P.tasks_rb, r = local - rb * P.tasks_rb;
                (void)rb;
                const int sp = r % P.splits;
                const int nk_all = P.K / CBK;
                const int nk = (sp + 1) * nk_all / P.splits - sp * nk_all / P.splits;
                const int acc = lt & 1;
                if (!mbar_wait(&tempty[acc], ((lt >> 1) & 1) ^ 1)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * CBN);
                for (int j = 0; j < nk; ++j, ++it) {
                    const int s = it % C_ST;
                    if (!mbar_wait(&full[s], (it / C_ST) & 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint8_t* st = smem + s * C_STAGE;
                    const uint64_t ad = sdesc_k_sw128(st);
                    const uint64_t bd = sdesc_k_sw128(st + 2 * C_A_TILE);
#pragma unroll
                    for (int kk = 0; kk < CBK / 16; ++kk) tc_mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (j | kk) != 0);
                    if (P.a_split) {
                        const uint64_t al = sdesc_k_sw128(st + C_A_TILE);
#pragma unroll
                        for (int kk = 0; kk < CBK / 16; ++kk) tc_mma_bf16(d, al + 2 * kk, bd + 2 * kk, idesc, 1u);
                    }
                    tc_commit(&empty[s]);
                }
                if (!ok) break;
                tc_commit(&tfull[acc]);
                ++lt;
            }
            if (!ok) fail(c);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;                      // 0 .. 7
        const int quarter = warp & 3, half = ew >> 2;  // TMEM lanes 32 quarter .., columns 32 half ..
        const int rloc = quarter * 32 + lane;
        float* stage = reinterpret_cast<float*>(smem + C_OFF_STAGING) + ew * EPI_STAGE_FLOATS;
        TaskSeq ts;
        ts.init(ph, n_rb);
        int lt = 0;
        bool ok = true;
        for (int g = blockIdx.x; ok && ts.seek(g, ph, n_ph, n_rb); g += G) {
            const ChainPhase& P = ph[ts.p];
            const int local = g - ts.start, rb = local / P.tasks_rb, r = local - rb * P.tasks_rb;
            if (P.op == CH_LN) {
                if (ts.p > 0) {
                    if (ew == 0 && lane == 0)
                        *last_flag = wait_count(c.cnt + (ts.p - 1) * CH_MAX_RB + rb, ph[ts.p - 1].done_rb, c);
                    epi_bar();
                    if (!*last_flag) { ok = false; break; }
                    epi_bar();  // every warp has read the flag
                }
                const int r0 = rb * CBM + r * CH_LN_ROWS;
                for (int i = ew; i < CH_LN_ROWS; i += C_EPI_WARPS) {
                    const int row = r0 + i;
                    if (row >= M) break;
                    if (P.D == 512) ln_row_task<16>(P, row);
                    else ln_row_task<32>(P, row);
                }
                epi_bar();
                if (ew == 0 && lane == 0) {
                    __threadfence();
                    atomicAdd(c.cnt + ts.p * CH_MAX_RB + rb, 1);
                }
                continue;
            }
            // GEMM tile
            const int tile = r / P.splits, sp = r - tile * P.splits;
            const int m0 = rb * CBM, n0 = tile * CBN;
            const int acc = lt & 1;
            if (!epi_all(mbar_wait(&tfull[acc], (lt >> 1) & 1))) { ok = false; break; }
            ++lt;
            tc_fence_after();
            const int c0 = half * 32;
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * CBN + c0), v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);  // this warp's TMEM reads are done
            const int row = m0 + rloc;
            if (P.splits > 1) {
                const long long tix = (long long)rb * P.tiles_n + tile;
                float* part = c.ws + P.ws_off + ((tix * P.splits + sp) * CBM + rloc) * CBN + c0;
                float4* p4 = reinterpret_cast<float4*>(part);
#pragma unroll
                for (int i = 0; i < 8; ++i) p4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                epi_bar();
                if (ew == 0 && lane == 0) {
                    __threadfence();
                    int* tc = c.tcnt + P.tc_off + tix;
                    const int old = atomicAdd(tc, 1);
                    const int last = old == P.splits - 1;
                    if (last) atomicExch(tc, 0);  // ready for the next launch
                    *last_flag = last;
                }
                epi_bar();
                const int last = *last_flag;
                epi_bar();  // every warp has read the flag before it is written again
                if (!last) continue;
                __threadfence();
                float sum[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) sum[i] = 0.f;
                for (int q = 0; q < P.splits; ++q) {
                    if (q == sp) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) sum[i] += v[i];
                    } else {
                        const float4* o4 = reinterpret_cast<const float4*>(
                            c.ws + P.ws_off + ((tix * P.splits + q) * CBM + rloc) * CBN + c0);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 t = __ldcg(o4 + i);
                            sum[4 * i] += t.x; sum[4 * i + 1] += t.y; sum[4 * i + 2] += t.z; sum[4 * i + 3] += t.w;
                        }
                    }
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = sum[i];
            }
            run_epilogue(P.ep, row, M, n0 + c0, v, stage);
            epi_bar();
            if (ew == 0 && lane == 0) {
                __threadfence();
                atomicAdd(c.cnt + ts.p * CH_MAX_RB + rb, 1);
            }
        }
        if (!ok) {
            if (lane == 0) fail(c);
        }
    }
    __syncwarp();
    // leave: the last CTA out zeroes the completion counters for the next launch
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, 2 * CBN);
    if (threadIdx.x == 0) {
        __threadfence();
        const int old = atomicAdd(c.done, 1);
        if (old == G - 1) {
            for (int i = 0; i < n_ph * CH_MAX_RB; ++i) c.cnt[i] = 0;
            *c.done = 0;
            *c.abort = 0;
            __threadfence();
        }
    }
}

int chain_smem_bytes() { return C_SMEM; }

cudaError_t launch_chain(const ChainPhase* d_phases, int n_phases, int M, const ChainCtl& ctl, int grid,
                         cudaStream_t s) {
    if (n_phases < 1 || n_phases > CH_MAX_PHASES || M < 1 || (M + CBM - 1) / CBM > CH_MAX_RB || grid < 1)
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C_SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C_THREADS);
    cfg.dynamicSmemBytes = C_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chain_kernel, d_phases, n_phases, M, ctl);
}

}  // namespace cac
