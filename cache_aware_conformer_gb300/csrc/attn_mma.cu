// Rectangular rel-pos attention of a streaming step on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation).
//
// Work unit: one (stream, head) with nq <= 4 new queries at absolute
// positions p0 .. p0 + nq - 1 and the Nk = Lc + nq <= 80 keys p0 - Lc .. p0 +
// nq - 1 (cache + new rows of the stream's K/V rings).  One warp per unit:
//
//   ac[j][i] = K[j] . (q_i + u)      A = K rows (16 keys per tile),   B = q + u
//   bd[r][i] = P[r] . (q_i + v)      A = position-table rows r,       B = q + v
//   score[i][j] = (ac[j][i] + bd[p_i - p_j - rmin][i]) * scale, masked to the
//                 query's key window, softmax over j
//   out[i][d]   = sum_j prob[i][j] V[j][d]      A = V^T (ldmatrix.trans),  B = prob
//
// The queries and the probabilities are fp32; each enters the MMA as a split
// pair (hi = bf16(x), lo = bf16(x - hi)) occupying two of the eight B columns
// (columns 0..3: hi of queries 0..3, columns 4..7: lo), so one MMA per tile
// carries them at ~16 significant bits and hi + lo is recombined from the
// fp32 accumulators with one shuffle.  K, V and the position table are bf16
// already (exact operands).
//
// Staging: TMA tensor copies with the 128-byte swizzle (chunk c of row r at
// chunk position c ^ (r & 7)), so the ldmatrix row reads are conflict-free.
// One copy brings a whole ring (R <= 80 rows, in slot order) of one stream,
// layer and head; logical key j lives in row (s0 + j) mod R, which each lane
// folds into its ldmatrix row address (rows R .. 79 stay zero).  Ring rows
// that hold no key of this step (logical j >= Nk) are masked in the softmax,
// and their V rows are zeroed in shared memory before probs @ V.  The position table (weights, rows
// r >= NR zeroed) is copied before the wait on the previous kernel, the rings
// after it, by one producer thread that runs up to AW_STAGES units ahead of
// the consumer warps (persistent blocks, one per SM).
#include <algorithm>
#include <cfloat>

#include "kernels.cuh"

namespace cac {

namespace {
constexpr int AM_ROWS = 80;                      // key / rel rows per unit (5 tiles of 16)
constexpr int AM_ROWB = 128;                     // bytes per row (64 bf16)
constexpr int AM_MAT = AM_ROWS * AM_ROWB;        // one [80][64] bf16 matrix
constexpr int AM_SLD = 84;                       // fp32 row stride of the score arrays
constexpr int AW_CONS = 8;                       // consumer warps per block
constexpr int AW_STAGES = 8;                     // ring stages, one unit's K and V rows each
constexpr int AW_THREADS = 32 * (1 + AW_CONS);
constexpr int AW_STAGE = 2 * AM_MAT;
constexpr int AW_SCORES = 2 * 4 * AM_SLD * 4;    // per consumer: [4][AM_SLD] ac / probs + bd / output
constexpr int AW_OFF_RING = AM_MAT;              // after the position table
constexpr int AW_OFF_SC = AW_OFF_RING + AW_STAGES * AW_STAGE;
constexpr int AW_OFF_BAR = AW_OFF_SC + AW_CONS * AW_SCORES;
constexpr int AW_SMEM = AW_OFF_BAR + (2 * AW_STAGES + 1) * 8 + 1024 /*alignment slack*/;
static_assert(AW_SMEM <= 227 * 1024, "shared memory");

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return (uint32_t)(row * AM_ROWB + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D += A * B, m16n8k16, bf16 in, fp32 accumulate
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// half 0: bf16(x); half 1: bf16(x - bf16(x))
__device__ __forceinline__ bf16 split_part(float x, int half) {
    const bf16 hi = __float2bfloat16_rn(x);
    return half ? __float2bfloat16_rn(x - __bfloat162float(hi)) : hi;
}
__device__ __forceinline__ uint32_t pack2(bf16 lo16, bf16 hi16) {
    return (uint32_t)__bfloat16_as_ushort(lo16) | ((uint32_t)__bfloat16_as_ushort(hi16) << 16);
}

// ac or bd for the five 16-row tiles of one [80][64] matrix against the
// split-query B fragments; result rows (keys / rels) x queries into S[i][row].
// Shared row of logical row j of a ring of R rows copied in slot order
// starting at slot s0: (s0 + j) mod R for j < R, else j (a zero row).
__device__ __forceinline__ int ring_row(int j, int s0, int R) {
    if (j >= R) return j;
    j += s0;
    return j >= R ? j - R : j;
}

__device__ __forceinline__ void score_tiles(uint32_t mat, int s0, int R, const uint32_t (&b)[4][2], float* S,
                                            int lane) {
    const int g = lane >> 2, c = lane & 3;
#pragma unroll
    for (int mt = 0; mt < AM_ROWS / 16; ++mt) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int row = ring_row(mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3), s0, R);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            uint32_t a[4];
            ldsm_x4(mat + swz(row, ks * 2 + (lane >> 4)), a);
            mma16816(acc, a, b[ks][0], b[ks][1]);
        }
        // columns 2c, 2c+1 (c < 2: hi of queries 2c, 2c+1; c >= 2: their lo)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], 2);
        if (c < 2) {
            const int r0 = mt * 16 + g;
            S[(2 * c) * AM_SLD + r0] = acc[0];
            S[(2 * c + 1) * AM_SLD + r0] = acc[1];
            S[(2 * c) * AM_SLD + r0 + 8] = acc[2];
            S[(2 * c + 1) * AM_SLD + r0 + 8] = acc[3];
        }
    }
}

__device__ __forceinline__ float wmax(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float wsum(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ void mbar_arrive_local(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// One unit's scores, softmax and probs @ V (the consumer side).  Km / Vm: the
// unit's K and V rows in shared memory; bu / bv: the split-query B fragments.
__device__ __forceinline__ void attend_unit(const AttnParams& a, uint32_t Pm, uint32_t Km, uint32_t Vm, int s0,
                                            const uint32_t (&bu)[4][2], const uint32_t (&bv)[4][2], float* Sac,
                                            float* Sbd, int p0, int Lc, int nq, int lane, float (&acc)[4][4]) {
    const int g = lane >> 2, c = lane & 3;
    const int Nk = Lc + nq;
    score_tiles(Km, s0, a.R, bu, Sac, lane);
    score_tiles(Pm, 0, AM_ROWS, bv, Sbd, lane);
    __syncwarp();
    // masked softmax per query over its key window (absolute positions)
    const int kpos0 = p0 - Lc;
    for (int i = 0; i < nq; ++i) {
        const int pq = p0 + i;
        int lo, hi;
        if (a.rc > 0) {
            lo = max(pq - a.left, 0);
            hi = pq + a.rc;
        } else {
            const int cc = (pq / a.chunk) * a.chunk;
            lo = max(cc - a.left, 0);
            hi = cc + a.chunk - 1;
        }
        float sv[3];
        float m = -FLT_MAX;
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            const int j = lane + 32 * t, pk = kpos0 + j;
            const bool ok = j < Nk && pk >= lo && pk <= hi;
            sv[t] = ok ? (Sac[i * AM_SLD + j] + Sbd[i * AM_SLD + (pq - pk - a.rmin)]) * a.scale : -FLT_MAX;
            m = fmaxf(m, sv[t]);
        }
        m = wmax(m);
        float sum = 0.f;
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            sv[t] = sv[t] == -FLT_MAX ? 0.f : __expf(sv[t] - m);
            sum += sv[t];
        }
        sum = wsum(sum);
        const float inv = 1.f / sum;
#pragma unroll
        for (int t = 0; t < 3; ++t) {
            const int j = lane + 32 * t;
            if (j < AM_ROWS) Sac[i * AM_SLD + j] = sv[t] * inv;
        }
    }
    __syncwarp();
    // out^T[d][col] = V^T[d][:] . prob^T[:][col]; B column g -> query g & 3, half g >> 2
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[mt][k] = 0.f;
    const int qi = g & 3, half = g >> 2;
    const bool has = qi < nq;
#pragma unroll
    for (int ks = 0; ks < AM_ROWS / 16; ++ks) {
        uint32_t bp[2];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int j = ks * 16 + 2 * c + 8 * hh;
            const float p0v = has ? Sac[qi * AM_SLD + j] : 0.f;
            const float p1v = has ? Sac[qi * AM_SLD + j + 1] : 0.f;
            bp[hh] = pack2(split_part(p0v, half), split_part(p1v, half));
        }
        const int key = ring_row(ks * 16 + (lane & 7) + ((lane >> 4) << 3), s0, a.R);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            uint32_t av[4];
            ldsm_x4_t(Vm + swz(key, mt * 2 + ((lane >> 3) & 1)), av);
            mma16816(acc[mt], av, bp[0], bp[1]);
        }
    }
}

// Split-query B fragments: column g -> query g & 3, half g >> 2; rows (dims)
// 16 ks + 2c, +1 and 16 ks + 2c + 8, +9.
__device__ __forceinline__ void query_frags(const AttnParams& a, const float* q, int h, int nq, int lane,
                                            uint32_t (&bu)[4][2], uint32_t (&bv)[4][2]) {
    constexpr int HD = 64;
    const int g = lane >> 2, c = lane & 3;
    const int qi = g & 3, half = g >> 2;
    const bool has = qi < nq;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int d = ks * 16 + 2 * c + 8 * hh;
            float2 qq = make_float2(0.f, 0.f);
            if (has) qq = *reinterpret_cast<const float2*>(q + (long long)qi * a.ldq + d);
            const float2 uu = __ldg(reinterpret_cast<const float2*>(a.pbu + h * HD + d));
            const float2 vv = __ldg(reinterpret_cast<const float2*>(a.pbv + h * HD + d));
            bu[ks][hh] = has ? pack2(split_part(qq.x + uu.x, half), split_part(qq.y + uu.y, half)) : 0u;
            bv[ks][hh] = has ? pack2(split_part(qq.x + vv.x, half), split_part(qq.y + vv.y, half)) : 0u;
        }
    }
}

// Persistent, warp-specialized: block (x, h) serves the streams b = x, x +
// gridDim.x, ... of head h.  Warp 0 lane 0 produces: per unit it waits for a
// free ring stage and issues the TMA copies of the unit's K and V rings into
// it.  Warps 1..AW_CONS consume units round-robin (consumer w takes units w-1,
// w-1+AW_CONS, ...; unit k lives in stage k mod AW_STAGES), loading their query
// fragments before waiting for the stage.
__global__ void __launch_bounds__(AW_THREADS, 1)
    attn_stream_ws_kernel(const __grid_constant__ AttnMaps tm, AttnParams a, int* status) {
    extern __shared__ uint8_t sm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    const int h = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t Pm = sbase;
    const uint32_t ring = sbase + AW_OFF_RING;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + AW_OFF_BAR);
    uint64_t* empty = full + AW_STAGES;
    uint64_t* pbar = empty + AW_STAGES;
    constexpr int HD = 64;

    // position table rows NR .. AM_ROWS-1 are zero (rel values no key reaches),
    // and so are the ring rows R .. AM_ROWS-1 of every stage (no copy writes them)
    for (int e = threadIdx.x; e < (AM_ROWS - a.NR) * 8; e += blockDim.x) {
        const int r = a.NR + (e >> 3);
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(Pm + swz(r, e & 7)), "r"(0) : "memory");
    }
    {
        const int per = (AM_ROWS - a.R) * 8;  // 16-byte chunks per matrix
        for (int e = threadIdx.x; e < 2 * AW_STAGES * per; e += blockDim.x) {
            const int mtx = e / per, r = a.R + (e % per >> 3);
            const uint32_t base = sbase + AW_OFF_RING + mtx * AM_MAT;  // stage st: matrices 2 st (K), 2 st + 1 (V)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(base + swz(r, e & 7)), "r"(0) : "memory");
        }
    }
    if (threadIdx.x == 0) {
        for (int st = 0; st < AW_STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], 1);
        }
        mbar_init(pbar, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm.k);
        tma_prefetch_desc(&tm.v);
        // weights: before the wait on the previous kernel
        mbar_expect_tx(pbar, (uint32_t)a.NR * AM_ROWB);
        tma_load_3d(sm, &tm.p, 0, 0, h, pbar);
    }
    __syncthreads();
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            for (int k = 0;; ++k) {
                const int b = blockIdx.x + k * gridDim.x;
                if (b >= a.nb) break;
                const int st = k % AW_STAGES;
                if (!mbar_wait(&empty[st], ((k / AW_STAGES) & 1) ^ 1)) {
                    latch_error(status, CAC_E_TIMEOUT);
                    break;
                }
                int id = a.ids[b];
                if (!in_range(id, a.n_streams, status)) id = 0;  // checked build: latched, stay in bounds
                const int blk = (id * a.L + a.layer) * a.H + h;
                uint8_t* Ks = sm + AW_OFF_RING + st * AW_STAGE;
                mbar_expect_tx(&full[st], 2u * a.R * AM_ROWB);
                tma_load_3d(Ks, &tm.k, 0, 0, blk, &full[st]);
                tma_load_3d(Ks + AM_MAT, &tm.v, 0, 0, blk, &full[st]);
            }
        }
        return;
    }

    const int cw = warp - 1;
    float* Sac = reinterpret_cast<float*>(sm + AW_OFF_SC + cw * AW_SCORES);  // ac, then probabilities
    float* Sbd = Sac + 4 * AM_SLD;                                          // bd, then the output rows
    const int nq = a.nq;
    const int g = lane >> 2, c = lane & 3;
    bool table = false;
    for (int k = cw;; k += AW_CONS) {
        const int b = blockIdx.x + k * gridDim.x;
        if (b >= a.nb) break;
        const int st = k % AW_STAGES;
        int id = a.ids[b];
        if (!in_range(id, a.n_streams, status)) id = 0;  // checked build: latched, stay in bounds
        int p0 = a.pos[id];
        if (!in_range(p0, 1 << 30, status)) p0 = 0;
        const int Lc = min(p0, a.left);
        if (!in_range(Lc + nq - 1, a.R, status)) break;   // more keys than ring rows
        const int s0 = (p0 - Lc) % a.R;
        uint32_t bu[4][2], bv[4][2];
        query_frags(a, a.q + (long long)b * nq * a.ldq + h * HD, h, nq, lane, bu, bv);
        if (!table) {
            if (!mbar_wait(pbar, 0)) {
                if (lane == 0) latch_error(status, CAC_E_TIMEOUT);
                break;
            }
            table = true;
        }
        if (!mbar_wait(&full[st], (k / AW_STAGES) & 1)) {
            if (lane == 0) latch_error(status, CAC_E_TIMEOUT);
            break;
        }
        const uint32_t Km = ring + st * AW_STAGE, Vm = Km + AM_MAT;
        // V rows that hold no key of this step enter probs @ V with probability
        // 0: make them zero, whatever the ring slot held
        for (int e = lane; e < (a.R - (Lc + nq)) * 8; e += 32) {
            const int r = ring_row(Lc + nq + (e >> 3), s0, a.R);
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(Vm + swz(r, e & 7)), "r"(0) : "memory");
        }
        __syncwarp();
        float acc[4][4];
        attend_unit(a, Pm, Km, Vm, s0, bu, bv, Sac, Sbd, p0, Lc, nq, lane, acc);
        fence_proxy_async_smem();  // the zeroed V rows before the next TMA copy into this stage
        __syncwarp();
        if (lane == 0) mbar_arrive_local(&empty[st]);  // the stage's last shared-memory access is done
        // recombine hi + lo, stage out[i][d] (fp32) in Sbd, then write the rows
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) acc[mt][q4] += __shfl_xor_sync(0xffffffffu, acc[mt][q4], 2);
        float* O = Sbd;
        if (c < 2) {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int d = mt * 16 + g;
                O[(2 * c) * 64 + d] = acc[mt][0];
                O[(2 * c + 1) * 64 + d] = acc[mt][1];
                O[(2 * c) * 64 + d + 8] = acc[mt][2];
                O[(2 * c + 1) * 64 + d + 8] = acc[mt][3];
            }
        }
        __syncwarp();
        bf16* dst = static_cast<bf16*>(a.out) + (long long)b * nq * a.ldo + h * HD;
        for (int i = 0; i < nq; ++i) {
            const float2 o = *reinterpret_cast<const float2*>(O + i * 64 + 2 * lane);
            const __nv_bfloat162 hi2 = __floats2bfloat162_rn(o.x, o.y);
            bf16* row = dst + (long long)i * a.ldo + 2 * lane;
            *reinterpret_cast<__nv_bfloat162*>(row) = hi2;
            if (a.out_split > 0) {
                const float2 hf = __bfloat1622float2(hi2);
                *reinterpret_cast<__nv_bfloat162*>(row + a.out_split) =
                    __floats2bfloat162_rn(o.x - hf.x, o.y - hf.y);
            }
        }
        __syncwarp();  // the output staging is read before the next unit's bd scores overwrite it
    }
    pdl_trigger();
}
// Offline encode, chunked mask: block (h, sequence) stages the sequence's K
// and V rows of head h once (one TMA copy each) plus the head's position
// table; AO_WARPS warps take the sequence's query chunks round-robin.  A chunk
// of nq <= chunk queries at q0 (a multiple of chunk) sees the keys klo =
// max(q0 - left, 0) .. q0 + nq - 1: the streaming unit with Lc = q0 - klo whose
// logical key j sits in shared row klo + j.  Its score tiles read the 80 rows
// klo .. klo + 79, so the staged block holds ao_rows(T, left) >= T + 79 - left
// rows; rows from the sequence length on are zeroed (their probabilities are
// 0, and 0 * V must stay 0).
constexpr int AO_WARPS = 8;
constexpr int AO_THREADS = 32 * AO_WARPS;

__host__ __device__ constexpr int ao_rows(int T, int left) {
    return ((T + 80 - left > AM_ROWS ? T + 80 - left : AM_ROWS) + 15) / 16 * 16;
}
inline size_t ao_smem(int rows) {
    return 1024 /*align*/ + AM_MAT + 2 * (size_t)rows * AM_ROWB + (size_t)AO_WARPS * AW_SCORES + 2 * 8;
}

__global__ void __launch_bounds__(AO_THREADS)
    attn_offline_mma_kernel(const __grid_constant__ AttnMaps tm, AttnParams a, int* status) {
    extern __shared__ uint8_t sm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    const int h = blockIdx.x, seq = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows = ao_rows(a.T, a.left);
    const uint32_t sbase = smem_u32(sm);
    const uint32_t Pm = sbase, Km = sbase + AM_MAT, Vm = Km + rows * AM_ROWB;
    float* scores = reinterpret_cast<float*>(sm + AM_MAT + 2 * rows * AM_ROWB);
    uint64_t* bar = reinterpret_cast<uint64_t*>(scores + AO_WARPS * AW_SCORES / 4);  // [0] table, [1] K/V
    constexpr int HD = 64;

    for (int e = threadIdx.x; e < (AM_ROWS - a.NR) * 8; e += blockDim.x)
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(Pm + swz(a.NR + (e >> 3), e & 7)), "r"(0)
                     : "memory");
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
        mbar_expect_tx(&bar[0], (uint32_t)a.NR * AM_ROWB);
        tma_load_3d(sm, &tm.p, 0, 0, h, &bar[0]);  // weights: before the wait on the previous kernel
    }
    __syncthreads();
    pdl_wait();
    if (threadIdx.x == 0) {
        mbar_expect_tx(&bar[1], 2u * rows * AM_ROWB);
        tma_load_2d(sm + AM_MAT, &tm.k, h * HD, seq * a.T, &bar[1]);
        tma_load_2d(sm + AM_MAT + rows * AM_ROWB, &tm.v, h * HD, seq * a.T, &bar[1]);
    }
    const int len = a.seq_len[seq];
    const bool landed = mbar_wait(&bar[0], 0) && mbar_wait(&bar[1], 0);
    if (!__syncthreads_and(landed)) {
        if (threadIdx.x == 0) latch_error(status, CAC_E_TIMEOUT);
        return;
    }
    for (int e = threadIdx.x; e < (rows - len) * 8; e += blockDim.x) {
        const int r = len + (e >> 3);
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(Km + swz(r, e & 7)), "r"(0) : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(Vm + swz(r, e & 7)), "r"(0) : "memory");
    }
    __syncthreads();

    AttnParams ao = a;
    ao.R = 1 << 20;  // no ring: logical key j of a chunk at shared row klo + j
    float* Sac = scores + warp * (AW_SCORES / 4);
    float* Sbd = Sac + 4 * AM_SLD;
    const int g = lane >> 2, c = lane & 3;
    const long long rb = (long long)seq * a.T;
    for (int u = warp; u * a.chunk < len; u += AO_WARPS) {
        const int q0 = u * a.chunk, nq = min(a.chunk, len - q0);
        const int klo = max(q0 - a.left, 0), Lc = q0 - klo;
        uint32_t bu[4][2], bv[4][2];
        query_frags(a, a.q + (rb + q0) * a.ldq + h * HD, h, nq, lane, bu, bv);
        float acc[4][4];
        attend_unit(ao, Pm, Km, Vm, klo, bu, bv, Sac, Sbd, q0, Lc, nq, lane, acc);
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) acc[mt][q4] += __shfl_xor_sync(0xffffffffu, acc[mt][q4], 2);
        float* O = Sbd;
        if (c < 2) {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const int d = mt * 16 + g;
                O[(2 * c) * 64 + d] = acc[mt][0];
                O[(2 * c + 1) * 64 + d] = acc[mt][1];
                O[(2 * c) * 64 + d + 8] = acc[mt][2];
                O[(2 * c + 1) * 64 + d + 8] = acc[mt][3];
            }
        }
        __syncwarp();
        bf16* dst = static_cast<bf16*>(a.out) + (rb + q0) * a.ldo + h * HD;
        for (int i = 0; i < nq; ++i) {
            const float2 o = *reinterpret_cast<const float2*>(O + i * 64 + 2 * lane);
            const __nv_bfloat162 hi2 = __floats2bfloat162_rn(o.x, o.y);
            bf16* row = dst + (long long)i * a.ldo + 2 * lane;
            *reinterpret_cast<__nv_bfloat162*>(row) = hi2;
            if (a.out_split > 0) {
                const float2 hf = __bfloat1622float2(hi2);
                *reinterpret_cast<__nv_bfloat162*>(row + a.out_split) =
                    __floats2bfloat162_rn(o.x - hf.x, o.y - hf.y);
            }
        }
        __syncwarp();  // the output staging is read before the next chunk's bd scores overwrite it
    }
    pdl_trigger();
}

}  // namespace

bool attention_stream_mma_ok(const AttnParams& a, int act_bf16) {
    return act_bf16 && a.maps && a.HD == 64 && a.R <= AM_ROWS && a.R >= a.left + a.nq && a.nq >= 1 && a.nq <= 4 &&
           a.left + a.nq <= AM_ROWS && a.NR <= AM_ROWS && a.rmin <= 0 && a.ldq % 2 == 0 && a.ldo % 2 == 0 &&
           a.out_split % 2 == 0;
}

bool attention_offline_mma_ok(const AttnParams& a, int act_bf16) {
    // keys of a chunk: q0 - left .. q0 + chunk - 1 (<= 80 rows); rel = p_q - p_k in
    // -(chunk - 1) .. left + chunk - 1 must index the table rows 0 .. NR - 1 < 80
    return act_bf16 && a.maps && a.HD == 64 && a.rc == 0 && a.chunk >= 1 && a.chunk <= 4 && a.left >= 0 &&
           a.left + a.chunk <= AM_ROWS && a.NR <= AM_ROWS && a.rmin <= -(a.chunk - 1) &&
           a.left + a.chunk - 1 - a.rmin < a.NR && a.T >= 1 && ao_rows(a.T, a.left) <= 256 &&
           ao_smem(ao_rows(a.T, a.left)) <= 227 * 1024 && a.ldq % 2 == 0 && a.ldo % 2 == 0 && a.out_split % 2 == 0;
}

int attention_offline_box_rows(int T, int left) { return ao_rows(T, left); }

cudaError_t launch_attention_offline_mma(const AttnParams& a, int* status, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attn_offline_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    return launch_k(attn_offline_mma_kernel, dim3(a.H, a.nb), dim3(AO_THREADS), ao_smem(ao_rows(a.T, a.left)), s, 1,
                    *a.maps, a, status);
}

cudaError_t launch_attention_stream_mma(const AttnParams& a, int* status, cudaStream_t s) {
    static bool attr = false;
    static int sms = 0;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attn_stream_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             AW_SMEM);
        if (e != cudaSuccess) return e;
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        attr = true;
    }
    // one block per SM in total: the heads split the SMs, each block serves a strided share of the streams
    const int per_head = std::max(1, std::min((a.nb + AW_CONS - 1) / AW_CONS, sms / std::max(1, a.H)));
    dim3 grid(per_head, a.H);
    return launch_k(attn_stream_ws_kernel, grid, dim3(AW_THREADS), AW_SMEM, s, 1, *a.maps, a, status);
}

}  // namespace cac
