// Host engine of the cache-aware Conformer library: weight upload, per-stream
// GPU-resident state pools, the step planner that turns one push of many
// streams into a fixed sequence of kernel launches (optionally replayed from a
// CUDA graph), flush, the offline chunked-causal encode, state export/import,
// and the extern "C" entry points declared in include/cac.h.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "../../include/cac_ops.h"
#include "chain.cuh"
#include "gemm.cuh"
#include "kernels.cuh"
#include "status.cuh"

using namespace cac;

namespace {

constexpr int MEL = 128;
constexpr int TAIL = 14;
constexpr int CONV_CACHE = 8;
constexpr int N_TAPS = 7;  // per-layer trace taps; tap 7 = subsampled input

uint16_t f2bf(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
float bf2f(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

#define CK(call)                                                                          \
    do {                                                                                  \
        cudaError_t e_ = (call);                                                          \
        if (e_ != cudaSuccess) {                                                          \
            std::fprintf(stderr, "cac: %s failed: %s\n", #call, cudaGetErrorString(e_)); \
            return CAC_E_CUDA;                                                            \
        }                                                                                 \
    } while (0)

#define RET(call)                    \
    do {                             \
        int r_ = (call);             \
        if (r_ != CAC_OK) return r_; \
    } while (0)

struct Lin {
    void* w = nullptr;   // [N][K] bf16 or fp32
    float* b = nullptr;  // [N] or null
    int N = 0, K = 0;
    int BN = 128;
    CUtensorMap tm;      // bf16 weights on the tcgen05 path (BN-row boxes)
    CUtensorMap tm128;   // the same with 128-row boxes (persistent GEMM), when N % 128 == 0
    bool has128 = false;
    // palette form (cac_model_create_palette): 6-bit indices [N][3K/4] bytes and
    // one 64-entry bf16 table per 64-row block of the outputs
    bool pal = false;
    void* packed = nullptr;
    uint16_t* ptab = nullptr;
    CUtensorMap tmp;     // packed indices, 48-byte x 64-row boxes
};

struct LayerW {
    float *ff1_g = nullptr, *ff1_b = nullptr, *att_g = nullptr, *att_b = nullptr, *conv_g = nullptr,
          *conv_b = nullptr, *ff2_g = nullptr, *ff2_b = nullptr, *out_g = nullptr, *out_b = nullptr;
    Lin ff1_w1, ff1_w2, qkv, wo, pw1, pw2, ff2_w1, ff2_w2;
    void* Ppad = nullptr;  // attention position table [H][NR][HD], activation dtype
    CUtensorMap Pmap;      // bf16, HD 64: one copy = one head's table (NR rows)
    bool has_pmap = false;
    // LayerNorm folded into the projection after it (fold_ln): bias b + W beta and
    // column sums sum_k gamma_k W[n][k] of the attention, conv and FF2 LayerNorms
    float *qkv_fb = nullptr, *pw1_fb = nullptr, *ff2_fb = nullptr;
    float *qkv_cs = nullptr, *pw1_cs = nullptr, *ff2_cs = nullptr;
    float *pbu = nullptr, *pbv = nullptr, *P = nullptr, *dwT = nullptr, *bdw = nullptr, *bng = nullptr,
          *bnb = nullptr;
};

struct OfflineWs {
    size_t bytes = 0;
    void* base = nullptr;
};

}  // namespace

struct cac_model {
    cac_config cfg{};
    int bf16 = 1, tc = 1;
    int split = 1;  // bf16: LayerNorm outputs enter their GEMMs as split (hi, lo) operands
    int split_ffh = 0;  // bf16, d_model >= 1024: the FF hidden activations enter the down-projection split too
    int fold_ln = 0;    // streaming steps: the attention, conv and FF2 LayerNorms run inside the GEMMs
    int sms = 152;      // streaming multiprocessors of the device
    int device = -1;    // the device current at creation: weights and pools live there
    int D = 0, H = 0, HD = 0, F = 0, L = 0, J = 0;
    int rmin = 0, NR = 0;
    std::vector<void*> allocs;
    Lin sub1, sub2, sub3, subo, joint;
    std::vector<LayerW> layers;
    int* status = nullptr;
    OfflineWs ws;
    long long launches = 0;
    struct ChainRec* rec = nullptr;  // set while a pool step records GEMM / LayerNorm phases into chains
};

namespace {

int dalloc(cac_model* m, size_t bytes, void** out) {
    void* p = nullptr;
    if (cudaMalloc(&p, std::max<size_t>(bytes, 16)) != cudaSuccess) return nomem();
    m->allocs.push_back(p);
    *out = p;
    return CAC_OK;
}

int upload_f32(cac_model* m, const float* src, size_t n, float** out) {
    void* p;
    RET(dalloc(m, n * sizeof(float), &p));
    CK(cudaMemcpy(p, src, n * sizeof(float), cudaMemcpyHostToDevice));
    *out = static_cast<float*>(p);
    return CAC_OK;
}

// Upload a [N][K] weight (rows optionally gathered through `perm`) and its bias.
int upload_lin(cac_model* m, const float* w, const float* b, int N, int K, Lin* lin, const std::vector<int>* perm) {
    lin->N = N;
    lin->K = K;
    const size_t n = (size_t)N * K;
    void* p;
    if (m->bf16) {
        std::vector<uint16_t> h(n);
        for (int r = 0; r < N; ++r) {
            const int src = perm ? (*perm)[r] : r;
            for (int k = 0; k < K; ++k) h[(size_t)r * K + k] = f2bf(w[(size_t)src * K + k]);
        }
        RET(dalloc(m, n * 2, &p));
        CK(cudaMemcpy(p, h.data(), n * 2, cudaMemcpyHostToDevice));
    } else {
        std::vector<float> h(n);
        for (int r = 0; r < N; ++r) {
            const int src = perm ? (*perm)[r] : r;
            std::memcpy(&h[(size_t)r * K], &w[(size_t)src * K], sizeof(float) * K);
        }
        RET(dalloc(m, n * 4, &p));
        CK(cudaMemcpy(p, h.data(), n * 4, cudaMemcpyHostToDevice));
    }
    lin->w = p;
    if (b) {
        std::vector<float> hb(N);
        for (int r = 0; r < N; ++r) hb[r] = b[perm ? (*perm)[r] : r];
        RET(upload_f32(m, hb.data(), N, &lin->b));
    }
    if (m->tc) {
        lin->BN = 64;  // 128 x 64 tiles: M = 512 rows already give 4 x N/64 CTAs
        if (N % lin->BN || K % 64) return CAC_E_UNSUPPORTED;
        if (!make_tmap_bf16(&lin->tm, p, K, N, (uint64_t)K * 2, lin->BN)) return CAC_E_CUDA;
        lin->has128 = N % 128 == 0;
        if (lin->has128 && !make_tmap_bf16(&lin->tm128, p, K, N, (uint64_t)K * 2, 128)) return CAC_E_CUDA;
    }
    return CAC_OK;
}

// Palette form of a projection for cac_model_create_palette: each weight's index
// in its matrix's 64-entry table (exact value match; the lowest index among
// equal entries; -0 and +0 alike), packed 6 bits per weight along K in the
// GEMM's row order (`perm` as in upload_lin), and one bf16 table per 64-row
// block of the outputs.  tab_of(src) is the table of source row src; the rows
// of a block must share one.  A weight absent from its table, or a table entry
// that is not a bf16 value, is CAC_E_INVAL.
template <class TabOf>
int pal_attach(cac_model* m, Lin* lin, const float* w, int N, int K, const std::vector<int>* perm, TabOf tab_of) {
    if (N % 64 || K % 64) return CAC_E_UNSUPPORTED;
    auto key = [](float v) {
        uint32_t b;
        std::memcpy(&b, &v, 4);
        return b == 0x80000000u ? 0u : b;
    };
    const size_t rb = (size_t)K * 6 / 8;
    std::vector<uint8_t> packed((size_t)N * rb, 0);
    std::vector<uint16_t> tabs((size_t)N);
    for (int blk = 0; blk < N / 64; ++blk) {
        const float* T = nullptr;
        for (int r = blk * 64; r < blk * 64 + 64; ++r) {
            const float* t = tab_of(perm ? (*perm)[r] : r);
            if (!t) return CAC_E_INVAL;
            if (T && t != T) return CAC_E_UNSUPPORTED;
            T = t;
        }
        std::unordered_map<uint32_t, int> idx_of;
        for (int i = 63; i >= 0; --i) {  // descending: the lowest index of equal entries wins
            if (bf2f(f2bf(T[i])) != T[i]) return CAC_E_INVAL;
            idx_of[key(T[i])] = i;
            tabs[(size_t)blk * 64 + i] = f2bf(T[i]);
        }
        for (int r = blk * 64; r < blk * 64 + 64; ++r) {
            const float* src = w + (size_t)(perm ? (*perm)[r] : r) * K;
            uint8_t* row = &packed[(size_t)r * rb];
            for (int k = 0; k < K; ++k) {
                const auto it = idx_of.find(key(src[k]));
                if (it == idx_of.end()) return CAC_E_INVAL;
                const uint32_t ix = (uint32_t)it->second;
                const int bit = 6 * k, off = bit & 7;
                row[bit >> 3] |= (uint8_t)(ix << off);
                if (off > 2) row[(bit >> 3) + 1] |= (uint8_t)(ix >> (8 - off));
            }
        }
    }
    void* pk;
    void* pt;
    RET(dalloc(m, packed.size(), &pk));
    RET(dalloc(m, tabs.size() * 2, &pt));
    CK(cudaMemcpy(pk, packed.data(), packed.size(), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(pt, tabs.data(), tabs.size() * 2, cudaMemcpyHostToDevice));
    if (!make_tmap_packed(&lin->tmp, pk, rb, (uint64_t)N)) return CAC_E_CUDA;
    lin->packed = pk;
    lin->ptab = static_cast<uint16_t*>(pt);
    lin->pal = true;
    return CAC_OK;
}

// Constants of a projection W (stored [N][K], bias b) that consumes LN(x) =
// gamma * z + beta with the LayerNorm folded into its GEMM: the GEMM's A operand
// is gamma * x (written by the producer of x), and
//   LN(x) W^T + b = rstd (sum_k gamma_k x_k W_k - mean colsum) + bias_f,
// colsum[n] = sum_k gamma_k W[n][k] over the stored (rounded) weights, bias_f[n]
// = b[n] + sum_k W[n][k] beta_k (fp64 on the host).  perm reorders the outputs
// as in upload_lin.
int upload_ln_fold(cac_model* m, const float* w, const float* b, const float* gamma, const float* beta, int N, int K,
                   const std::vector<int>* perm, float** bias_f, float** colsum) {
    std::vector<float> bf(N), cs(N);
    for (int r = 0; r < N; ++r) {
        const int src = perm ? (*perm)[r] : r;
        double acc_b = b[src], acc_c = 0.0;
        for (int k = 0; k < K; ++k) {
            const float wv = w[(size_t)src * K + k];
            acc_b += (double)wv * beta[k];
            acc_c += (double)gamma[k] * (m->bf16 ? (double)bf2f(f2bf(wv)) : (double)wv);
        }
        bf[r] = (float)acc_b;
        cs[r] = (float)acc_c;
    }
    RET(upload_f32(m, bf.data(), N, bias_f));
    return upload_f32(m, cs.data(), N, colsum);
}

struct Cursor {
    const float* p;
    size_t left;
    const float* take(size_t n) {
        if (n > left) return nullptr;
        const float* r = p;
        p += n;
        left -= n;
        return r;
    }
};

int validate(const cac_config* c) {
    if (!c) return CAC_E_INVAL;
    if (c->n_layers <= 0 || c->d_model <= 0 || c->n_heads <= 0 || c->ff_dim <= 0) return CAC_E_INVAL;
    if (c->d_model % c->n_heads) return CAC_E_INVAL;
    const int hd = c->d_model / c->n_heads;
    if (hd != 64 && hd != 16) return CAC_E_UNSUPPORTED;
    if (c->dw_kernel != 9 || c->mel_bins != MEL) return CAC_E_UNSUPPORTED;
    if (c->d_model % 64 || c->ff_dim % 64 || c->joint_dim % 64 || c->d_model > 1024) return CAC_E_UNSUPPORTED;
    if (c->att_left < 0 || c->att_chunk <= 0 || c->att_chunk > 8) return CAC_E_INVAL;
    if (c->dtype != CAC_DTYPE_F32 && c->dtype != CAC_DTYPE_BF16) return CAC_E_INVAL;
    if (c->right_context < 0 || c->right_context > 8) return CAC_E_UNSUPPORTED;
    if (c->right_context > 0 && (c->emit_frames <= 0 || c->lookahead_frames < 0 ||
                                 c->emit_frames + c->lookahead_frames > 24 ||
                                 c->att_left + c->emit_frames + c->lookahead_frames > 96))
        return CAC_E_UNSUPPORTED;
    if (c->right_context == 0 && c->att_left + 8 > 80) return CAC_E_UNSUPPORTED;
    return CAC_OK;
}

// Split-K policy knobs: CAC_SPLIT_TARGET (CTAs the split aims for, default
// 120) and CAC_SPLIT_MIN_SLICES (64-wide K slices each split keeps, default 8,
// at least 2), read once from the environment for tuning sweeps.
int env_int(const char* name, int dflt, int lo, int hi) {
    const char* e = std::getenv(name);
    if (!e || !*e) return dflt;
    const int v = std::atoi(e);
    return v < lo ? lo : (v > hi ? hi : v);
}

int choose_splits(int tiles, int nk) {
    // split K until the grid covers most of the 152 SMs, at most 4 ways and only
    // while every split keeps >= 8 K slices: below that the cluster reduction
    // costs more than the shorter main loop saves (measured at M = 512: K = 512
    // runs faster unsplit at every N of the encoder, K = 2048 fastest 4-way)
    static const int target = env_int("CAC_SPLIT_TARGET", 120, 1, 1 << 20);
    static const int min_slices = env_int("CAC_SPLIT_MIN_SLICES", 8, 2, 1 << 20);
    int splits = 1;
    while (splits < 4 && tiles * splits < target && nk / (splits + 1) >= min_slices) ++splits;
    return splits;
}

// ---------------------------------------------------------------------------
// chains: consecutive projections / LayerNorms of a step recorded as phases and
// run by one persistent launch (chain.cu) when something that cannot join the
// chain (an attention launch, the end of the step) comes next.
// ---------------------------------------------------------------------------
struct ChainKey {
    int nb, n, nvalid;
    const void *mel, *enc, *joint, *ids, *scratch;
    long long mel_bstride;
    int out_bstride, out_off, seq;
    bool operator<(const ChainKey& o) const {
        return std::tie(nb, n, nvalid, mel, enc, joint, ids, scratch, mel_bstride, out_bstride, out_off, seq) <
               std::tie(o.nb, o.n, o.nvalid, o.mel, o.enc, o.joint, o.ids, o.scratch, o.mel_bstride, o.out_bstride,
                        o.out_off, o.seq);
    }
};
struct ChainProg {
    ChainPhase* d = nullptr;  // device copy of the phases
    int n = 0;
    int M = 0;
};
}  // namespace

struct ChainRec {
    bool on = false;
    std::vector<ChainPhase> ph;  // phases recorded since the last flush
    int M = 0;
    ChainKey ctx{};              // the step being recorded (seq counts its flushes)
    std::map<ChainKey, ChainProg> cache;
    ChainCtl ctl;                // device counters and split-K workspace
    long long ws_floats = 0, tcnt_n = 0;
    int sms = 152;
    long long* launches = nullptr;
    cac_pool* pool = nullptr;    // for per-class timing of the chain launches
    bool recorded = false;       // the last GEMM call was recorded (profiling: no launch to time)
    void release() {
        for (auto& kv : cache)
            if (kv.second.d) cudaFree(kv.second.d);
        cache.clear();
    }
};

namespace {

// Split-K of a chained projection: enough tasks to cover most SMs (K ranges of
// at least two 64-wide slices, at most 4 splits).
int chain_splits(int tiles, int nk) {
    static const int max_s = env_int("CAC_CHAIN_MAX_SPLITS", 4, 1, 4);  // tuning knob
    int s = 1;
    while (s < max_s && tiles * s < 120 && nk / (s + 1) >= 2) ++s;
    return s;
}

int prof_begin(cac_pool* p, int cls, cudaStream_t s);
int prof_end(cac_pool* p, cudaStream_t s);

// Run the recorded phases as one chain launch (building and caching the
// device program on its first use; never while the stream is being captured).
int chain_flush(ChainRec* r, cudaStream_t s) {
    if (!r || r->ph.empty()) return CAC_OK;
    const int n_rb = (r->M + 127) / 128;
    ChainKey key = r->ctx;
    key.seq = r->ctx.seq++;
    auto it = r->cache.find(key);
    if (it == r->cache.end() || it->second.n != (int)r->ph.size() || it->second.M != r->M) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        CK(cudaStreamIsCapturing(s, &cs));
        if (cs != cudaStreamCaptureStatusNone) return CAC_E_STATE;  // programs are built by an eager run first
        if (r->cache.size() >= 512) {  // eager callers with ever-new buffers: start over
            CK(cudaStreamSynchronize(s));
            r->release();
        }
        long long ws = 0, tc = 0;
        for (ChainPhase& P : r->ph) {
            if (P.op == CH_GEMM && P.splits > 1) {
                P.ws_off = ws;
                ws += chain_ws_floats(P, n_rb);
                P.tc_off = (int)tc;
                tc += (long long)n_rb * P.tiles_n;
            }
        }
        if (ws > r->ws_floats) {
            CK(cudaStreamSynchronize(s));
            if (r->ctl.ws) cudaFree(r->ctl.ws);
            r->ctl.ws = nullptr;
            r->ws_floats = 0;
            if (cudaMalloc(&r->ctl.ws, sizeof(float) * ws) != cudaSuccess) return nomem();
            r->ws_floats = ws;
        }
        if (tc > r->tcnt_n) {
            CK(cudaStreamSynchronize(s));
            if (r->ctl.tcnt) cudaFree(r->ctl.tcnt);
            r->ctl.tcnt = nullptr;
            r->tcnt_n = 0;
            if (cudaMalloc(&r->ctl.tcnt, sizeof(int) * tc) != cudaSuccess) return nomem();
            CK(cudaMemset(r->ctl.tcnt, 0, sizeof(int) * tc));
            r->tcnt_n = tc;
        }
        ChainProg prog;
        prog.n = (int)r->ph.size();
        prog.M = r->M;
        if (cudaMalloc(&prog.d, sizeof(ChainPhase) * prog.n) != cudaSuccess) return nomem();
        CK(cudaMemcpy(prog.d, r->ph.data(), sizeof(ChainPhase) * prog.n, cudaMemcpyHostToDevice));
        if (it != r->cache.end() && it->second.d) {
            CK(cudaStreamSynchronize(s));
            cudaFree(it->second.d);
        }
        r->cache[key] = prog;
        it = r->cache.find(key);
    }
    if (r->pool) RET(prof_begin(r->pool, 15 /* chain */, s));
    CK(launch_chain(it->second.d, it->second.n, it->second.M, r->ctl, r->sms, s));
    if (r->pool) RET(prof_end(r->pool, s));
    if (r->launches) ++*r->launches;
    r->ph.clear();
    return CAC_OK;
}

// Record a LayerNorm (launch_layernorm's arguments, bf16 activations) as a
// chain phase; false when it cannot join a chain.
bool chain_record_ln(ChainRec* r, const float* x, int M, int D, const float* g1, const float* b1, float* y_f32,
                     void* y_act, const float* g2, const float* b2, void* z_act, int grp, int grp_stride,
                     int row_off, int split) {
    if (!r || !r->on || (D != 512 && D != 1024) || (!r->ph.empty() && r->M != M) ||
        (int)r->ph.size() >= CH_MAX_PHASES || (M + 127) / 128 > CH_MAX_RB)
        return false;
    ChainPhase P;
    std::memset(static_cast<void*>(&P), 0, sizeof(P));
    P.op = CH_LN;
    P.tasks_rb = 128 / CH_LN_ROWS;
    P.done_rb = P.tasks_rb;
    P.splits = 1;
    P.ep = EpiParams();
    P.x = x; P.g1 = g1; P.b1 = b1; P.g2 = g2; P.b2 = b2;
    P.y_f32 = y_f32;
    P.y_act = static_cast<bf16*>(y_act);
    P.z_act = static_cast<bf16*>(z_act);
    P.D = D; P.grp = grp; P.grp_stride = grp_stride; P.row_off = row_off; P.split = split;
    r->M = M;
    r->ph.push_back(P);
    return true;
}

// GEMM dispatch: tcgen05 for bf16 models (unless the SIMT debugging twin is
// requested), SIMT for fp32 models.  conv_C > 0: A is a stride-2 convolution
// window read through the im2col view (M output rows = window row pairs).
// a_split: A is a split operand (hi | lo, row stride lda >= 2K), see launch_layernorm.
int gemm(cac_model* m, const void* A, long long lda, int M, int K, const Lin& W, int conv_C, EpiParams ep,
         cudaStream_t s, long long* launches, int a_split = 0) {
    if (M <= 0) return CAC_OK;
    if (a_split && !conv_C && lda < 2LL * K) return CAC_E_INVAL;
    ep.act_bf16 = m->bf16;
    if (m->tc && m->rec && m->rec->on) {
        ChainRec* r = m->rec;
        const bool chainable = !conv_C && !W.pal && W.BN == 64 && W.N % 64 == 0 &&
                               (ep.kind == EPI_STORE || ep.kind == EPI_RESID || ep.kind == EPI_QKV ||
                                ep.kind == EPI_GLUDW) &&
                               (r->ph.empty() || r->M == M) && (int)r->ph.size() < CH_MAX_PHASES &&
                               (M + 127) / 128 <= CH_MAX_RB;
        if (chainable) {
            ChainPhase P;
            std::memset(static_cast<void*>(&P), 0, sizeof(P));
            if (!make_tmap_bf16(&P.ta, A, a_split ? 2 * K : K, M, (uint64_t)lda * 2, 128)) return CAC_E_CUDA;
            P.tb = W.tm;
            P.op = CH_GEMM;
            P.K = K;
            P.N = W.N;
            P.a_split = a_split ? 1 : 0;
            P.tiles_n = W.N / 64;
            P.splits = chain_splits(P.tiles_n * ((M + 127) / 128), K / 64);
            P.tasks_rb = P.tiles_n * P.splits;
            P.done_rb = P.tiles_n;
            P.ep = ep;
            r->M = M;
            r->ph.push_back(P);
            r->recorded = true;
            return CAC_OK;
        }
        RET(chain_flush(r, s));  // run what is pending before a launch that cannot join
    }
    if (m->tc) {
        CUtensorMap tmA;
        const bool ok = conv_C ? make_tmap_bf16_conv(&tmA, A, (uint64_t)conv_C * (a_split ? 2 : 1), (uint64_t)M + 1, 128)
                               : make_tmap_bf16(&tmA, A, a_split ? 2 * K : K, M, (uint64_t)lda * 2, 128);
        if (!ok) return CAC_E_CUDA;
        // many output tiles (the offline encode): the persistent kernel, whose
        // epilogue of one tile overlaps the main loop of the next
        if (W.has128 && !W.pal && ep.kind != EPI_GLUDW && (long long)((M + 127) / 128) * (W.N / 128) >= 2 * m->sms) {
            CK(launch_gemm_tc_persistent(&tmA, &W.tm128, M, W.N, K, conv_C, a_split, ep, m->status, s));
            ++*launches;
            return CAC_OK;
        }
        // long K (the FF down-projections): 128-column tiles split 4 ways over K,
        // each rank finishing one 32-column chunk (owner mode; CAC_SPLIT_OWNER=0
        // keeps 64-column tiles finished by rank 0)
        static const bool owner_on = env_int("CAC_SPLIT_OWNER", 1, 0, 1) != 0;
        static const int owner_min = env_int("CAC_SPLIT_OWNER_MIN_SLICES", 32, 4, 1 << 20);
        if (owner_on && W.has128 && !W.pal && !conv_C && ep.kind != EPI_GLUDW && K / 64 >= owner_min) {
            CK(launch_gemm_tc(&tmA, &W.tm128, M, W.N, K, 128, conv_C, 4, a_split, ep, m->status, s));
            ++*launches;
            return CAC_OK;
        }
        // the fused depthwise conv reads its stream's rows within one CTA: no split-K
        const int splits = ep.kind == EPI_GLUDW ? 1 : choose_splits((W.N / W.BN) * ((M + 127) / 128), K / 64);
        if (W.pal)  // palette weights: 64-row tiles decoded in the kernel
            CK(launch_gemm_tc(&tmA, &W.tmp, M, W.N, K, 64, conv_C, splits, a_split, ep, m->status, s, W.ptab));
        else
            CK(launch_gemm_tc(&tmA, &W.tm, M, W.N, K, W.BN, conv_C, splits, a_split, ep, m->status, s));
    } else {
        CK(launch_gemm_simt(m->bf16, A, lda, W.w, K, M, W.N, K, conv_C, a_split, ep, s));
    }
    ++*launches;
    return CAC_OK;
}

size_t act_bytes(const cac_model* m) { return m->bf16 ? 2 : 4; }

}  // namespace

// ===========================================================================
// model
// ===========================================================================
extern "C" size_t cac_weights_size(const cac_config* c) {
    const int v = validate(c);
    if (v != CAC_OK && v != CAC_E_UNSUPPORTED) return 0;
    const size_t D = c->d_model, F = c->ff_dim, M = c->mel_bins, J = c->joint_dim, K = c->dw_kernel;
    size_t n = D * 3 * M + D + 2 * (D * 3 * D + D) + D * D + D;
    const size_t ff = 2 * D + F * D + F + D * F + D;
    const size_t att = 2 * D + 4 * (D * D + D) + D * D + 2 * D;
    const size_t conv = 2 * D + 2 * D * D + 2 * D + D * K + D + 2 * D + D * D + D;
    n += (size_t)c->n_layers * (2 * ff + att + conv + 2 * D);
    n += J * D + J;
    return n;
}

namespace {
// The model from a dense weight blob; with `tables` (palette form, see
// cac_model_create_palette) the projections also take their palette form.
int model_create(const cac_config* cfg, const float* weights, size_t n_floats, const float* tables, cac_model** out) {
    if (!out || !weights) return CAC_E_INVAL;
    *out = nullptr;
    RET(validate(cfg));
    if (n_floats != cac_weights_size(cfg)) return CAC_E_INVAL;
    cac_model* m = new (std::nothrow) cac_model();
    if (!m) return CAC_E_NOMEM;
    m->cfg = *cfg;
    m->bf16 = cfg->dtype == CAC_DTYPE_BF16;
    m->tc = m->bf16 && !cfg->gemm_simt;
    m->split = m->bf16;
    m->split_ffh = m->bf16 && cfg->d_model >= 1024;
    m->fold_ln = m->bf16 && m->tc && cfg->d_model % 32 == 0;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) {
            m->device = dev;
            cudaDeviceGetAttribute(&m->sms, cudaDevAttrMultiProcessorCount, dev);
        }
    }
    m->D = cfg->d_model;
    m->H = cfg->n_heads;
    m->HD = m->D / m->H;
    m->F = cfg->ff_dim;
    m->L = cfg->n_layers;
    m->J = cfg->joint_dim;
    const int back = std::max(cfg->att_chunk - 1, cfg->right_context);
    m->rmin = -back;
    m->NR = cfg->att_left + std::max(cfg->att_chunk - 1, 0) - m->rmin + 1;
    const int D = m->D, F = m->F, H = m->H, HD = m->HD;

    auto fail = [&](int code) {
        cac_model_destroy(m);
        return code;
    };
    Cursor c{weights, n_floats};
    int r;
    void* st;
    if ((r = dalloc(m, sizeof(int), &st)) != CAC_OK) return fail(r);
    m->status = static_cast<int*>(st);
    if (cudaMemset(m->status, 0, sizeof(int)) != cudaSuccess) return fail(CAC_E_CUDA);

    const float *w, *b;
    // palette tables in their documented order (see cac_model_create_palette)
    auto table = [&](int i) -> const float* { return tables ? tables + (size_t)64 * i : nullptr; };
    auto palette = [&](Lin* dst, const float* ww, int N, int K, const std::vector<int>* perm, int ti) {
        if (!tables) return (int)CAC_OK;
        const float* t = table(ti);
        return pal_attach(m, dst, ww, N, K, perm, [t](int) { return t; });
    };
    w = c.take((size_t)D * 3 * MEL); b = c.take(D);
    if ((r = upload_lin(m, w, b, D, 3 * MEL, &m->sub1, nullptr)) != CAC_OK ||
        (r = palette(&m->sub1, w, D, 3 * MEL, nullptr, 0)) != CAC_OK)
        return fail(r);
    w = c.take((size_t)D * 3 * D); b = c.take(D);
    if ((r = upload_lin(m, w, b, D, 3 * D, &m->sub2, nullptr)) != CAC_OK ||
        (r = palette(&m->sub2, w, D, 3 * D, nullptr, 1)) != CAC_OK)
        return fail(r);
    w = c.take((size_t)D * 3 * D); b = c.take(D);
    if ((r = upload_lin(m, w, b, D, 3 * D, &m->sub3, nullptr)) != CAC_OK ||
        (r = palette(&m->sub3, w, D, 3 * D, nullptr, 2)) != CAC_OK)
        return fail(r);
    w = c.take((size_t)D * D); b = c.take(D);
    if ((r = upload_lin(m, w, b, D, D, &m->subo, nullptr)) != CAC_OK ||
        (r = palette(&m->subo, w, D, D, nullptr, 3)) != CAC_OK)
        return fail(r);

    // GLU interleave: every 32 output columns of pw1 = 16 value rows then their 16 gate rows
    std::vector<int> glu_perm(2 * D);
    for (int j = 0; j < 2 * D; ++j) {
        const int s = j / 32, q = j % 32;
        glu_perm[j] = q < 16 ? 16 * s + q : D + 16 * s + (q - 16);
    }

    // position table pe(r) for r = rmin .. rmin + NR - 1 (shared by all layers)
    float* pe = nullptr;
    {
        void* p;
        if ((r = dalloc(m, sizeof(float) * m->NR * D, &p)) != CAC_OK) return fail(r);
        pe = static_cast<float*>(p);
        if (launch_sinusoid(pe, m->NR, m->rmin, D, 0) != cudaSuccess) return fail(CAC_E_CUDA);
    }

    m->layers.resize(m->L);
    std::vector<float> tmp;
    for (int l = 0; l < m->L; ++l) {
        LayerW& Lw = m->layers[l];
        auto vec = [&](float** dst, size_t n) {
            const float* s = c.take(n);
            return s ? upload_f32(m, s, n, dst) : CAC_E_INVAL;
        };
        // the host copy of the last vec() upload (a LayerNorm's gamma / beta)
        const float* host_g = nullptr;
        const float* host_b = nullptr;
        auto vec_ln = [&](float** g, float** be) {
            host_g = c.take(D);
            host_b = c.take(D);
            if (!host_g || !host_b) return CAC_E_INVAL;
            int e = upload_f32(m, host_g, D, g);
            return e ? e : upload_f32(m, host_b, D, be);
        };
        // a projection that consumes the last vec_ln() LayerNorm; also stored folded (fold_ln)
        const int tl = 5 + 11 * l;  // this layer's first palette table
        auto lin = [&](Lin* dst, int N, int K, const std::vector<int>* perm, int ti, float** fold_b = nullptr,
                       float** colsum = nullptr) {
            const float* ww = c.take((size_t)N * K);
            const float* bb = c.take(N);
            if (!ww || !bb) return (int)CAC_E_INVAL;
            int e = upload_lin(m, ww, bb, N, K, dst, perm);
            if (e == CAC_OK && fold_b && m->fold_ln)
                e = upload_ln_fold(m, ww, bb, host_g, host_b, N, K, perm, fold_b, colsum);
            if (e == CAC_OK) e = palette(dst, ww, N, K, perm, tl + ti);
            return e;
        };
        if ((r = vec(&Lw.ff1_g, D)) || (r = vec(&Lw.ff1_b, D)) || (r = lin(&Lw.ff1_w1, F, D, nullptr, 0)) ||
            (r = lin(&Lw.ff1_w2, D, F, nullptr, 1)))
            return fail(r);
        if ((r = vec_ln(&Lw.att_g, &Lw.att_b))) return fail(r);
        {   // q, k, v concatenated into one [3D][D] projection
            const float *wq = c.take((size_t)D * D), *bq = c.take(D), *wk = c.take((size_t)D * D), *bk = c.take(D),
                        *wv = c.take((size_t)D * D), *bv = c.take(D);
            if (!wv || !bv) return fail(CAC_E_INVAL);
            std::vector<float> wqkv((size_t)3 * D * D), bqkv(3 * D);
            std::memcpy(&wqkv[0], wq, sizeof(float) * D * D);
            std::memcpy(&wqkv[(size_t)D * D], wk, sizeof(float) * D * D);
            std::memcpy(&wqkv[(size_t)2 * D * D], wv, sizeof(float) * D * D);
            std::memcpy(&bqkv[0], bq, sizeof(float) * D);
            std::memcpy(&bqkv[D], bk, sizeof(float) * D);
            std::memcpy(&bqkv[2 * D], bv, sizeof(float) * D);
            if ((r = upload_lin(m, wqkv.data(), bqkv.data(), 3 * D, D, &Lw.qkv, nullptr)) != CAC_OK) return fail(r);
            if (tables && (r = pal_attach(m, &Lw.qkv, wqkv.data(), 3 * D, D, nullptr,
                                          [&](int src) { return table(tl + 2 + src / D); })) != CAC_OK)
                return fail(r);
            if (m->fold_ln && (r = upload_ln_fold(m, wqkv.data(), bqkv.data(), host_g, host_b, 3 * D, D, nullptr,
                                                  &Lw.qkv_fb, &Lw.qkv_cs)) != CAC_OK)
                return fail(r);
        }
        if ((r = lin(&Lw.wo, D, D, nullptr, 5))) return fail(r);
        {   // P = pe @ wpos^T, computed once per layer in fp32
            const float* wpos = c.take((size_t)D * D);
            if (!wpos) return fail(CAC_E_INVAL);
            float* wpos_d;
            if ((r = upload_f32(m, wpos, (size_t)D * D, &wpos_d)) != CAC_OK) return fail(r);
            void* p;
            if ((r = dalloc(m, sizeof(float) * m->NR * D, &p)) != CAC_OK) return fail(r);
            Lw.P = static_cast<float*>(p);
            EpiParams ep;
            ep.kind = EPI_STORE;
            ep.act_bf16 = 0;
            ep.out_f32 = Lw.P;
            ep.ldo = D;
            if (launch_gemm_simt(0, pe, D, wpos_d, D, m->NR, D, D, 0, 0, ep, 0) != cudaSuccess) return fail(CAC_E_CUDA);
            // head-major copy [H][NR][HD] in the activation dtype: one bulk copy per
            // (block, head) in the attention kernels
            std::vector<float> hp((size_t)m->NR * D), pad((size_t)H * m->NR * HD, 0.f);
            if (cudaMemcpy(hp.data(), Lw.P, hp.size() * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
                return fail(CAC_E_CUDA);
            for (int hh = 0; hh < H; ++hh)
                for (int rr = 0; rr < m->NR; ++rr)
                    std::memcpy(&pad[((size_t)hh * m->NR + rr) * HD], &hp[(size_t)rr * D + hh * HD],
                                sizeof(float) * HD);
            if (m->bf16) {
                std::vector<uint16_t> hb(pad.size());
                for (size_t k = 0; k < pad.size(); ++k) hb[k] = f2bf(pad[k]);
                void* pp;
                if ((r = dalloc(m, hb.size() * 2, &pp)) != CAC_OK) return fail(r);
                if (cudaMemcpy(pp, hb.data(), hb.size() * 2, cudaMemcpyHostToDevice) != cudaSuccess)
                    return fail(CAC_E_CUDA);
                Lw.Ppad = pp;
                if (HD == 64 && m->NR <= 256) {
                    if (!make_tmap_bf16_blocks(&Lw.Pmap, pp, m->NR, H, (uint64_t)m->NR * HD * 2, m->NR))
                        return fail(CAC_E_CUDA);
                    Lw.has_pmap = true;
                }
            } else {
                float* pf;
                if ((r = upload_f32(m, pad.data(), pad.size(), &pf)) != CAC_OK) return fail(r);
                Lw.Ppad = pf;
            }
        }
        if ((r = vec(&Lw.pbu, (size_t)H * HD)) || (r = vec(&Lw.pbv, (size_t)H * HD))) return fail(r);
        if ((r = vec_ln(&Lw.conv_g, &Lw.conv_b)) || (r = lin(&Lw.pw1, 2 * D, D, &glu_perm, 7, &Lw.pw1_fb, &Lw.pw1_cs)))
            return fail(r);
        {   // depthwise [D][9] -> [9][D]
            const float* wdw = c.take((size_t)D * 9);
            if (!wdw) return fail(CAC_E_INVAL);
            tmp.assign((size_t)9 * D, 0.f);
            for (int ch = 0; ch < D; ++ch)
                for (int k = 0; k < 9; ++k) tmp[(size_t)k * D + ch] = wdw[(size_t)ch * 9 + k];
            if ((r = upload_f32(m, tmp.data(), tmp.size(), &Lw.dwT)) != CAC_OK) return fail(r);
        }
        if ((r = vec(&Lw.bdw, D)) || (r = vec(&Lw.bng, D)) || (r = vec(&Lw.bnb, D)) ||
            (r = lin(&Lw.pw2, D, D, nullptr, 8)))
            return fail(r);
        if ((r = vec_ln(&Lw.ff2_g, &Lw.ff2_b)) || (r = lin(&Lw.ff2_w1, F, D, nullptr, 9, &Lw.ff2_fb, &Lw.ff2_cs)) ||
            (r = lin(&Lw.ff2_w2, D, F, nullptr, 10)))
            return fail(r);
        if ((r = vec(&Lw.out_g, D)) || (r = vec(&Lw.out_b, D))) return fail(r);
    }
    {
        const float* wj = c.take((size_t)m->J * D);
        const float* bj = c.take(m->J);
        if (!wj || !bj) return fail(CAC_E_INVAL);
        if ((r = upload_lin(m, wj, bj, m->J, D, &m->joint, nullptr)) != CAC_OK ||
            (r = palette(&m->joint, wj, m->J, D, nullptr, 4)) != CAC_OK)
            return fail(r);
    }
    if (c.left != 0) return fail(CAC_E_INVAL);
    if (cudaDeviceSynchronize() != cudaSuccess) return fail(CAC_E_CUDA);
    *out = m;
    return CAC_OK;
}
}  // namespace

extern "C" int cac_model_create(const cac_config* cfg, const float* weights, size_t n_floats, cac_model** out) {
    return model_create(cfg, weights, n_floats, nullptr, out);
}

extern "C" int cac_model_create_palette(const cac_config* cfg, const float* weights, size_t n_floats,
                                        const float* tables, size_t n_tables, cac_model** out) {
    if (!cfg || !tables || !out) return CAC_E_INVAL;
    if (cfg->dtype != CAC_DTYPE_BF16 || cfg->gemm_simt) return CAC_E_UNSUPPORTED;
    if (n_tables != (size_t)64 * (5 + 11 * (size_t)cfg->n_layers)) return CAC_E_INVAL;
    return model_create(cfg, weights, n_floats, tables, out);
}

extern "C" void cac_model_destroy(cac_model* m) {
    if (!m) return;
    cudaDeviceSynchronize();
    for (void* p : m->allocs) cudaFree(p);
    if (m->ws.base) cudaFree(m->ws.base);
    delete m;
}

extern "C" int cac_model_check(cac_model* m) {
    if (!m) return CAC_E_INVAL;
    CK(cudaDeviceSynchronize());
    int st = 0;
    CK(cudaMemcpy(&st, m->status, sizeof(int), cudaMemcpyDeviceToHost));
    CK(cudaMemset(m->status, 0, sizeof(int)));
    return st;
}

// ===========================================================================
// pool
// ===========================================================================
namespace {
constexpr int ID_SLOTS = 8;

struct GraphKey {
    int nb, n, nvalid;
    const void *mel, *enc, *joint;
    long long mel_bstride;
    int out_bstride, out_off;
    const void* ids;  // batch slot -> stream id array (a sub-batch's slice)
    int group;        // scratch set
    bool operator<(const GraphKey& o) const {
        return std::tie(nb, n, nvalid, mel, enc, joint, mel_bstride, out_bstride, out_off, ids, group) <
               std::tie(o.nb, o.n, o.nvalid, o.mel, o.enc, o.joint, o.mel_bstride, o.out_bstride, o.out_off, o.ids,
                        o.group);
    }
};
struct GraphEntry {
    int seen = 0;
    cudaGraphExec_t exec = nullptr;
    long long kernels = 0;
};
}  // namespace

// Scratch of one step: activations and windows of its rows
struct Scratch {
    void *win1 = nullptr, *win2 = nullptr, *win3 = nullptr, *y3 = nullptr;
    float* x = nullptr;
    void *xln = nullptr, *h = nullptr, *o = nullptr, *glu = nullptr, *yc = nullptr;
    float* q = nullptr;
    float2* stats = nullptr;  // fold_ln: per-row partials (sum, centred sum of squares) of 32 columns of x
};
constexpr int MAX_GROUPS = 8;

struct cac_pool {
    cac_model* m = nullptr;
    int S = 0, nmax = 0, R = 0;
    std::vector<void*> allocs;
    // per-stream device state
    int* pos = nullptr;        // subsampled frames consumed
    float* tail = nullptr;     // [S][14][128] fp32
    std::vector<AttnMaps> amaps;  // per layer: K/V ring and position-table tensor maps (tensor-core attention)
    void* kring = nullptr;     // [S][L][H][R][HD]
    void* vring = nullptr;
    void* conv = nullptr;      // [S][L][8][D]
    // step scratch in use (one of sc[], see use_scratch)
    void *win1 = nullptr, *win2 = nullptr, *win3 = nullptr, *y3 = nullptr;
    float* x = nullptr;
    void *xln = nullptr, *h = nullptr, *o = nullptr, *glu = nullptr, *yc = nullptr;
    float* q = nullptr;
    float2* stats = nullptr;
    // A chunked step over many streams runs as up to `groups` concurrent
    // sub-batches of at most group_streams streams each, forked onto the pool's
    // own CUDA streams: independent kernel chains overlap one another's
    // per-kernel latency.  sc[0] holds all S streams (every other path uses it).
    std::vector<Scratch> sc;
    int groups = 1, group_streams = 0;
    cudaStream_t gs[MAX_GROUPS] = {};
    cudaEvent_t fork_ev = nullptr, join_ev[MAX_GROUPS] = {};
    int* ids_dev = nullptr;     // batch slot -> stream id for the current push
    int* rids_dev = nullptr;    // ids of the current reset
    int* nvalid_dev = nullptr;  // flush: valid mel frames per batch slot
    int* status = nullptr;
    // host mirrors
    std::vector<uint8_t> alive, finished;
    std::vector<int> pos_host;
    // pinned id staging ring
    int* pinned = nullptr;
    cudaEvent_t slot_ev[ID_SLOTS] = {};
    int slot = 0;
    // host buffers of a cac_stream_push_host call whose step runs as concurrent
    // sub-batches: each sub-batch copies its slice in and out on its own stream
    struct HostIO {
        const float* mel = nullptr;  // page-locked source of the mel rows
        float* enc = nullptr;        // page-locked destinations (nullptr: not wanted)
        float* joint = nullptr;
    } hio;
    bool hio_on = false;
    // staging for cac_stream_push_host
    float* h_mel = nullptr;
    float* d_mel = nullptr;
    float* h_out = nullptr;
    float* d_out = nullptr;
    size_t h_mel_cap = 0, h_out_cap = 0;
    // graphs, tracing, counters
    bool graphs = false;
    std::map<GraphKey, GraphEntry> gcache;
    bool trace = false;
    float* trace_buf = nullptr;  // [L][7][rows][D] + [rows][D]
    int trace_rows = 0;
    long long launches = 0;
    long long ring_sstride = 0, conv_sstride = 0;
    size_t tail_elems = 0;
    // provisional tail (right_context > 0): frames subsampled vs emitted
    int* sub_pos = nullptr;     // [S] frames subsampled so far (pos = frames emitted)
    float* x0 = nullptr;        // [S][XC][D] exact subsampled frames not yet emitted
    int XC = 0;
    int* pids_dev = nullptr;    // stream ids of the current pass
    int* pmap_dev = nullptr;    // pass slot -> batch slot of the call
    std::vector<int> sub_host;
    std::vector<char*> guards;   // guard zones around the per-stream pools (palloc_guarded)
    // chains of projection / LayerNorm phases (chunked steps on the tcgen05 path)
    ChainRec chain;
    bool chains = false;  // cac_pool_set_chains (off by default: measured slower, see chain.cu)
    int cur_group = 0;   // scratch set in use
    // per-kernel-class CUDA-event timing (eager launches only)
    bool prof = false;
    std::vector<cudaEvent_t> ev;          // event pool, reused after each read
    std::vector<std::pair<int, int>> rec; // (class, index of the start event; end = start + 1)
    int prof_cls = -1;
};

namespace {

// A per-stream pool between two guard zones of GUARD_BYTES filled with 0xFF
// bytes (NaN in bf16 and fp32), checked by cac_pool_check_guards.
constexpr size_t GUARD_BYTES = 4096;
int palloc_guarded(cac_pool* p, size_t bytes, void** out) {
    char* d = nullptr;
    const size_t total = bytes + 2 * GUARD_BYTES;
    if (cudaMalloc(&d, total) != cudaSuccess) return nomem();
    p->allocs.push_back(d);
    if (cudaMemset(d, 0, total) != cudaSuccess || cudaMemset(d, 0xFF, GUARD_BYTES) != cudaSuccess ||
        cudaMemset(d + GUARD_BYTES + bytes, 0xFF, GUARD_BYTES) != cudaSuccess)
        return CAC_E_CUDA;
    p->guards.push_back(d);
    p->guards.push_back(d + GUARD_BYTES + bytes);
    *out = d + GUARD_BYTES;
    return CAC_OK;
}

int palloc(cac_pool* p, size_t bytes, void** out, bool zero = true) {
    void* d = nullptr;
    if (cudaMalloc(&d, std::max<size_t>(bytes, 16)) != cudaSuccess) return nomem();
    p->allocs.push_back(d);
    if (zero && cudaMemset(d, 0, std::max<size_t>(bytes, 16)) != cudaSuccess) return CAC_E_CUDA;
    *out = d;
    return CAC_OK;
}

// Make scratch set g the one the step functions use.
void use_scratch(cac_pool* p, int g) {
    const Scratch& sc = p->sc[g];
    p->cur_group = g;
    p->win1 = sc.win1; p->win2 = sc.win2; p->win3 = sc.win3; p->y3 = sc.y3;
    p->x = sc.x; p->xln = sc.xln; p->h = sc.h; p->o = sc.o; p->glu = sc.glu; p->yc = sc.yc; p->q = sc.q;
    p->stats = sc.stats;
}

// Copy `n` ids into the next pinned slot and queue their upload to `dst`.
int upload_ids(cac_pool* p, const int* ids, int n, int* dst, cudaStream_t s) {
    const int k = p->slot;
    p->slot = (p->slot + 1) % ID_SLOTS;
    CK(cudaEventSynchronize(p->slot_ev[k]));
    int* h = p->pinned + (size_t)k * p->S;
    std::memcpy(h, ids, sizeof(int) * n);
    CK(cudaMemcpyAsync(dst, h, sizeof(int) * n, cudaMemcpyHostToDevice, s));
    CK(cudaEventRecord(p->slot_ev[k], s));
    return CAC_OK;
}

int check_ids(cac_pool* p, int n, const int* ids, bool need_unfinished) {
    if (n <= 0 || n > p->S || !ids) return CAC_E_INVAL;
    std::vector<uint8_t> seen(p->S, 0);
    for (int i = 0; i < n; ++i) {
        const int id = ids[i];
        if (id < 0 || id >= p->S || seen[id]) return CAC_E_INVAL;
        seen[id] = 1;
        if (!p->alive[id]) return CAC_E_STATE;
        if (need_unfinished && p->finished[id]) return CAC_E_STATE;
    }
    return CAC_OK;
}

// split: src is a bf16 split operand [rows][2D]; the tap records hi + lo.
int trace_tap(cac_pool* p, int layer, int tap, const void* src, bool src_act, int rows, cudaStream_t s,
              bool split = false) {
    if (!p->trace) return CAC_OK;
    cac_model* m = p->m;
    const long long per = (long long)p->trace_rows * m->D;
    float* dst = tap == N_TAPS ? p->trace_buf + (long long)m->L * N_TAPS * per
                               : p->trace_buf + ((long long)layer * N_TAPS + tap) * per;
    if (split)
        CK(launch_split_to_f32(src, dst, rows, m->D, s));
    else
        CK(launch_to_f32(src, dst, (long long)rows * m->D, src_act && m->bf16, s));
    ++p->launches;
    return CAC_OK;
}

const char* const PROF_NAMES[] = {"stage_mel", "gemm_subsample", "gemm_sub_out", "layernorm",
                                  "gemm_ff_up", "gemm_ff_down", "gemm_qkv", "attention", "gemm_out_proj",
                                  "gemm_pw1_glu", "dwconv", "gemm_pw2", "gemm_joint", "advance", "reset",
                                  "chain"};
constexpr int N_PROF = 16;
enum { P_STAGE, P_SUB, P_SUBOUT, P_LN, P_FFUP, P_FFDOWN, P_QKV, P_ATT, P_OUT, P_PW1, P_DW, P_PW2, P_JOINT,
       P_ADV, P_RESET, P_CHAIN };

// Open a timed region of class `cls` on stream s (no-op unless profiling).
int prof_begin(cac_pool* p, int cls, cudaStream_t s) {
    if (!p->prof) return CAC_OK;
    const size_t need = 2 * (p->rec.size() + 1);
    while (p->ev.size() < need) {
        cudaEvent_t e;
        CK(cudaEventCreate(&e));
        p->ev.push_back(e);
    }
    const int i = (int)(2 * p->rec.size());
    p->rec.push_back({cls, i});
    p->chain.recorded = false;
    CK(cudaEventRecord(p->ev[i], s));
    return CAC_OK;
}
int prof_end(cac_pool* p, cudaStream_t s) {
    if (!p->prof) return CAC_OK;
    if (p->chain.recorded) {  // nothing launched: a GEMM recorded into a chain
        p->rec.pop_back();
        return CAC_OK;
    }
    CK(cudaEventRecord(p->ev[p->rec.back().second + 1], s));
    return CAC_OK;
}
#define PB(cls) RET(prof_begin(p, cls, s))
#define PE() RET(prof_end(p, s))

// Subsampling of n new frames for nb slots (ids[b]; the first new frame of
// stream id sits at posS[id]) into p->x rows [b * n + i].
//   mel: stream b's first mel row at mel + b * mel_bstride (8n rows; with
//        nvalid, rows >= nvalid[b] read as zero)
int run_subsample(cac_pool* p, int nb, int n, const float* mel, long long mel_bstride, const int* nvalid,
                  const int* ids, const int* posS, cudaStream_t s) {
    cac_model* m = p->m;
    const int D = m->D;
    const int M = nb * n;
    long long* lc = &p->launches;
    const int bf = m->bf16, sp = m->split;
    const int rwm = MEL * (1 + sp), rwd = D * (1 + sp);  // window row widths (split: hi | lo)

    // 1. mel staging: [melTail | mel] windows, tail update
    PB(P_STAGE);
    CK(launch_stage_mel(mel, mel_bstride, nvalid, p->win1, p->tail, ids, posS, n, nb, bf, sp, p->status, s, p->S));
    PE();
    ++*lc;
    // 2. three stride-2 convolutions (implicit GEMMs over the windows) + out linear
    const int W1 = TAIL + 8 * n, W2 = 4 * n + 6, W3 = 2 * n + 2;
    {
        EpiParams ep;
        ep.kind = EPI_SUB;
        ep.bias = m->sub1.b;
        ep.out_act = p->win2;
        ep.ldo = rwd;
        ep.split_out = sp ? D : 0;
        ep.ids = ids;
        ep.pos = posS;
        ep.n_streams = p->S;
        ep.status = p->status;
        ep.P = W1 / 2; ep.T_out = W2; ep.dst_rows = W2; ep.dst_off = 0; ep.tmult = 4; ep.toff = 6;
        PB(P_SUB);
        RET(gemm(m, p->win1, 2 * rwm, nb * (W1 / 2), 3 * MEL, m->sub1, MEL, ep, s, lc, sp));
        PE();
        ep.bias = m->sub2.b;
        ep.out_act = p->win3;
        ep.P = W2 / 2; ep.T_out = W3; ep.dst_rows = W3; ep.tmult = 2; ep.toff = 2;
        PB(P_SUB);
        RET(gemm(m, p->win2, 2 * rwd, nb * (W2 / 2), 3 * D, m->sub2, D, ep, s, lc, sp));
        PE();
        ep.bias = m->sub3.b;
        ep.out_act = p->y3;
        ep.P = W3 / 2; ep.T_out = n; ep.dst_rows = n; ep.tmult = 1; ep.toff = 0;
        PB(P_SUB);
        RET(gemm(m, p->win3, 2 * rwd, nb * (W3 / 2), 3 * D, m->sub3, D, ep, s, lc, sp));
        PE();
    }
    {
        EpiParams ep;
        ep.kind = EPI_STORE;
        ep.bias = m->subo.b;
        ep.out_f32 = p->x;
        ep.ldo = D;
        PB(P_SUBOUT);
        RET(gemm(m, p->y3, rwd, M, D, m->subo, 0, ep, s, lc, sp));
        PE();
    }
    RET(trace_tap(p, 0, N_TAPS, p->x, false, M, s));
    return CAC_OK;
}

// The layer stack over nq rows per slot (p->x rows [b * nq + i], queries at
// absolute positions pos[ids[b]] + i).  K/V rows of all nq frames go to the
// rings; the conv cache commits the first n_commit GLU rows.  The last
// ln_out writes enc (row remap b * out_bstride + out_off + i) or, when enc is
// null, p->x in place; its activation-dtype copy always lands in p->xln.
int run_layers(cac_pool* p, int nb, int nq, int n_commit, const int* ids, float* enc, int out_bstride, int out_off,
               cudaStream_t s) {
    cac_model* m = p->m;
    const int D = m->D, F = m->F, L = m->L;
    const int M = nb * nq, n = nq;
    long long* lc = &p->launches;
    const size_t ab = act_bytes(m);
    const int bf = m->bf16, sp = m->split;
    const long long ldl = sp ? 2LL * D : D;  // row stride of the split LayerNorm outputs in xln
    const int shf = m->split_ffh;
    const long long ldh = shf ? 2LL * F : F;  // row stride of the FF hidden activations (split: hi | lo)
    // fold_ln: the residual GEMM before the attention, conv and FF2 LayerNorms
    // writes the split operand of x into xln and its row partials into stats;
    // the GEMM after it applies the LayerNorm in its epilogue
    const bool fold = m->fold_ln && sp && p->stats;
    auto emit_split = [&](EpiParams& e, const float* gamma) {
        if (!fold) return;
        e.xs = static_cast<bf16*>(p->xln); e.ldxs = ldl; e.xs_lo = D; e.xs_gamma = gamma;
        e.stats_out = p->stats; e.stats_parts = D / 32;
    };
    auto use_fold = [&](EpiParams& e, const float* colsum) {
        e.ln_stats = p->stats; e.ln_colsum = colsum; e.ln_parts = D / 32; e.ln_rows = M;
    };
    // a LayerNorm launch, or a chain phase while the step records chains
    auto layernorm = [&](const float* x, const float* g1, const float* b1, float* y_f32, void* y_act,
                         const float* g2, const float* b2, void* z_act, int grp, int grp_stride, int row_off,
                         int split) -> int {
        if (chain_record_ln(m->rec, x, M, D, g1, b1, y_f32, y_act, g2, b2, z_act, grp, grp_stride, row_off, split))
            return CAC_OK;
        RET(chain_flush(m->rec, s));
        PB(P_LN);
        CK(launch_layernorm(x, M, D, g1, b1, y_f32, y_act, g2, b2, z_act, bf, grp, grp_stride, row_off, split, s));
        PE();
        ++*lc;
        return CAC_OK;
    };
    RET(layernorm(p->x, m->layers[0].ff1_g, m->layers[0].ff1_b, nullptr, p->xln, nullptr, nullptr, nullptr, 1 << 30,
                  0, 0, sp));

    for (int l = 0; l < L; ++l) {
        const LayerW& Lw = m->layers[l];
        EpiParams ep;
        // FF1: x += 1/2 * (W2 SiLU(W1 LN(x) + b1) + b2)   (LN(x) already in xln)
        ep.kind = EPI_STORE; ep.act = ACT_SILU; ep.bias = Lw.ff1_w1.b; ep.out_act = p->h; ep.ldo = ldh; ep.split_out = shf ? F : 0;
        PB(P_FFUP);
        RET(gemm(m, p->xln, ldl, M, D, Lw.ff1_w1, 0, ep, s, lc, sp));
        PE();
        ep = EpiParams(); ep.kind = EPI_RESID; ep.bias = Lw.ff1_w2.b; ep.x = p->x; ep.ldx = D; ep.scale = 0.5f;
        emit_split(ep, Lw.att_g);
        PB(P_FFDOWN);
        RET(gemm(m, p->h, ldh, M, F, Lw.ff1_w2, 0, ep, s, lc, shf));
        PE();
        RET(trace_tap(p, l, 0, p->x, false, M, s));
        // attention: xln = LN(x); Q and K/V into the rings
        if (!fold) {
            PB(P_LN);
            CK(launch_layernorm(p->x, M, D, Lw.att_g, Lw.att_b, nullptr, p->xln, nullptr, nullptr, nullptr, bf,
                                1 << 30, 0, 0, sp, s));
            PE();
            ++*lc;
        }
        ep = EpiParams(); ep.kind = EPI_QKV; ep.bias = fold ? Lw.qkv_fb : Lw.qkv.b; ep.D = D; ep.HD = m->HD; ep.R = p->R;
        if (fold) use_fold(ep, Lw.qkv_cs);
        ep.ring_sstride = p->ring_sstride;
        ep.kring = static_cast<char*>(p->kring) + (long long)l * m->H * p->R * m->HD * ab;
        ep.vring = static_cast<char*>(p->vring) + (long long)l * m->H * p->R * m->HD * ab;
        ep.q = p->q; ep.ldq = D; ep.ids = ids; ep.pos = p->pos; ep.nq = n;
        ep.n_streams = p->S; ep.status = p->status;
        PB(P_QKV);
        RET(gemm(m, p->xln, ldl, M, D, Lw.qkv, 0, ep, s, lc, sp));
        PE();
        {
            AttnParams a;
            a.q = p->q; a.ldq = D;
            a.k = ep.kring; a.v = ep.vring; a.sstride = p->ring_sstride; a.R = p->R;
            a.ids = ids; a.pos = p->pos; a.nq = n; a.n_streams = p->S;
            a.P = Lw.Ppad; a.rmin = m->rmin; a.NR = m->NR; a.pbu = Lw.pbu; a.pbv = Lw.pbv;
            a.out = p->o; a.ldo = (int)ldl; a.out_split = sp ? D : 0;
            a.H = m->H; a.D = D; a.HD = m->HD;
            a.left = m->cfg.att_left; a.chunk = m->cfg.att_chunk; a.rc = m->cfg.right_context;
            a.nb = nb;
            a.scale = 1.f / std::sqrt((float)m->HD);
            if (!p->amaps.empty()) { a.maps = &p->amaps[l]; a.layer = l; a.L = L; }
            RET(chain_flush(m->rec, s));  // the projections before attention run first
            PB(P_ATT);
            CK(launch_attention_stream(a, bf, p->status, s));
            PE();
            ++*lc;
        }
        RET(trace_tap(p, l, 1, p->o, true, M, s, sp));
        ep = EpiParams(); ep.kind = EPI_RESID; ep.bias = Lw.wo.b; ep.x = p->x; ep.ldx = D; ep.scale = 1.f;
        emit_split(ep, Lw.conv_g);
        PB(P_OUT);
        RET(gemm(m, p->o, ldl, M, D, Lw.wo, 0, ep, s, lc, sp));
        PE();
        RET(trace_tap(p, l, 2, p->x, false, M, s));
        // conv module
        if (!fold) {
            PB(P_LN);
            CK(launch_layernorm(p->x, M, D, Lw.conv_g, Lw.conv_b, nullptr, p->xln, nullptr, nullptr, nullptr, bf,
                                1 << 30, 0, 0, sp, s));
            PE();
            ++*lc;
        }
        void* conv_l = static_cast<char*>(p->conv) + (long long)l * CONV_CACHE * D * ab;
        // tcgen05 path, chunked steps whose frames per stream divide a warp: the
        // depthwise conv runs in the pw1 + GLU epilogue (a stream's rows share a warp)
        const bool fuse_dw = m->tc && sp && 32 % n == 0 && n_commit == n;
        ep = EpiParams(); ep.kind = fuse_dw ? EPI_GLUDW : EPI_GLU; ep.bias = fold ? Lw.pw1_fb : Lw.pw1.b;
        ep.out_act = p->glu; ep.ldo = D;
        if (fold) use_fold(ep, Lw.pw1_cs);
        if (fuse_dw) {
            ep.D = D; ep.nq = n; ep.ids = ids; ep.pos = p->pos;
            ep.n_streams = p->S; ep.status = p->status;
            ep.dw_ring = conv_l; ep.dw_sstride = p->conv_sstride;
            ep.dw_wT = Lw.dwT; ep.dw_bias = Lw.bdw; ep.dw_gamma = Lw.bng; ep.dw_beta = Lw.bnb; ep.dw_out = p->yc;
            ep.dw_rows = M;
        }
        PB(P_PW1);
        RET(gemm(m, p->xln, ldl, M, D, Lw.pw1, 0, ep, s, lc, sp));
        PE();
        RET(trace_tap(p, l, 3, p->glu, true, M, s));
        if (!fuse_dw) {
            PB(P_DW);
            CK(launch_dwconv(p->glu, conv_l, p->conv_sstride, ids, p->pos, n, n_commit, Lw.dwT, Lw.bdw, Lw.bng,
                             Lw.bnb, p->yc, D, nb, bf, s, p->S, p->status));
            PE();
            ++*lc;
        }
        RET(trace_tap(p, l, 4, p->yc, true, M, s));
        ep = EpiParams(); ep.kind = EPI_RESID; ep.bias = Lw.pw2.b; ep.x = p->x; ep.ldx = D; ep.scale = 1.f;
        emit_split(ep, Lw.ff2_g);
        PB(P_PW2);
        RET(gemm(m, p->yc, D, M, D, Lw.pw2, 0, ep, s, lc));
        PE();
        RET(trace_tap(p, l, 5, p->x, false, M, s));
        // FF2
        if (!fold) {
            PB(P_LN);
            CK(launch_layernorm(p->x, M, D, Lw.ff2_g, Lw.ff2_b, nullptr, p->xln, nullptr, nullptr, nullptr, bf,
                                1 << 30, 0, 0, sp, s));
            PE();
            ++*lc;
        }
        ep = EpiParams(); ep.kind = EPI_STORE; ep.act = ACT_SILU; ep.bias = fold ? Lw.ff2_fb : Lw.ff2_w1.b;
        ep.out_act = p->h; ep.ldo = ldh; ep.split_out = shf ? F : 0;
        if (fold) use_fold(ep, Lw.ff2_cs);
        PB(P_FFUP);
        RET(gemm(m, p->xln, ldl, M, D, Lw.ff2_w1, 0, ep, s, lc, sp));
        PE();
        ep = EpiParams(); ep.kind = EPI_RESID; ep.bias = Lw.ff2_w2.b; ep.x = p->x; ep.ldx = D; ep.scale = 0.5f;
        PB(P_FFDOWN);
        RET(gemm(m, p->h, ldh, M, F, Lw.ff2_w2, 0, ep, s, lc, shf));
        PE();
        // ln_out, fused with the next layer's FF1 LayerNorm (or, after the last
        // layer, writing the encoder frames to the caller and the joint input)
        if (l + 1 < L) {
            RET(layernorm(p->x, Lw.out_g, Lw.out_b, p->x, nullptr, m->layers[l + 1].ff1_g, m->layers[l + 1].ff1_b,
                          p->xln, 1 << 30, 0, 0, sp));
            RET(trace_tap(p, l, 6, p->x, false, M, s));
        } else {
            RET(layernorm(p->x, Lw.out_g, Lw.out_b, enc ? enc : p->x, p->xln, nullptr, nullptr, nullptr,
                          enc ? n : 1 << 30, enc ? out_bstride : 0, enc ? out_off : 0, 0));
            RET(trace_tap(p, l, 6, p->xln, true, M, s));
        }
    }
    return CAC_OK;
}

// Joint projection of the rows of act (activation dtype, grp rows per slot)
// into joint rows g' * out_bstride + out_off + i, g' = map ? map[g] : g.
int run_joint(cac_pool* p, const void* act, int M, int grp, float* joint, int out_bstride, int out_off,
              const int* map, cudaStream_t s) {
    cac_model* m = p->m;
    EpiParams ep;
    ep.kind = EPI_STORE;
    ep.bias = m->joint.b;
    ep.out_f32 = joint;
    ep.ldo = m->J;
    ep.grp = grp; ep.grp_stride = out_bstride; ep.row_off = out_off; ep.grp_map = map;
    PB(P_JOINT);
    RET(gemm(m, act, m->D, M, m->D, m->joint, 0, ep, s, &p->launches));
    PE();
    return CAC_OK;
}

// Whether a chunked step runs its projections and LayerNorms as chains: the
// pool asked for them (cac_pool_set_chains, or CAC_CHAIN=1 in the environment
// for every pool), the tcgen05 path with the folded LayerNorms and the fused
// depthwise conv, and no tracing.
bool chain_env() {
    static const bool on = [] {
        const char* e = std::getenv("CAC_CHAIN");
        return e && e[0] == '1';
    }();
    return on;
}
bool chain_step_ok(const cac_pool* p, int nb, int n) {
    const cac_model* m = p->m;
    return (p->chains || chain_env()) && m->tc && m->fold_ln && m->split && p->stats && 32 % n == 0 && !p->trace &&
           (m->D == 512 || m->D == 1024) && (nb * n + 127) / 128 <= CH_MAX_RB &&
           p->chain.ctl.cnt != nullptr;
}

// One chunked-causal step: nb batch slots (ids in p->ids_dev), n new frames each.
//   enc/joint: frame i of slot b goes to row b * out_bstride + out_off + i
int run_step(cac_pool* p, int nb, int n, const float* mel, long long mel_bstride, const int* nvalid, float* enc,
             float* joint, int out_bstride, int out_off, cudaStream_t s, const int* ids = nullptr) {
    if (!ids) ids = p->ids_dev;
    cac_model* m = p->m;
    const bool chained = chain_step_ok(p, nb, n);
    if (chained) {
        ChainRec& r = p->chain;
        r.on = true;
        r.ph.clear();
        r.ctx = ChainKey{nb, n, nvalid ? 1 : 0, mel, enc, joint, ids, p->x, mel_bstride, out_bstride, out_off, 0};
        r.launches = &p->launches;
        m->rec = &r;
    }
    int rc = run_subsample(p, nb, n, mel, mel_bstride, nvalid, ids, p->pos, s);
    if (rc == CAC_OK) rc = run_layers(p, nb, n, n, ids, enc, out_bstride, out_off, s);
    if (rc == CAC_OK && joint) rc = run_joint(p, p->xln, nb * n, n, joint, out_bstride, out_off, nullptr, s);
    if (chained) {
        if (rc == CAC_OK) rc = chain_flush(&p->chain, s);
        p->chain.on = false;
        p->chain.ph.clear();
        m->rec = nullptr;
    }
    RET(rc);
    PB(P_ADV);
    CK(launch_advance(p->pos, ids, nb, n, s, p->S, p->status));
    PE();
    ++p->launches;
    return CAC_OK;
}

// Provisional tail, one pass over the nbp streams in p->pids_dev: P frames
// from the x0 ring starting at the first unemitted one; E of them are emitted,
// frame i of batch slot k to enc/joint row p->pmap_dev[k] + i; K/V and the conv
// tail of the emitted frames are committed (the other P - E rows are
// recomputed by the next pass).
int run_pass(cac_pool* p, int nbp, int P, int E, float* enc, float* joint, cudaStream_t s) {
    cac_model* m = p->m;
    const int D = m->D;
    CK(launch_x0_gather(p->x0, p->x, p->pids_dev, p->pos, nbp, P, p->XC, D, s, p->S, p->status));
    ++p->launches;
    RET(run_layers(p, nbp, P, E, p->pids_dev, nullptr, 0, 0, s));
    // compact the emitted rows: fp32 frames to the caller, activation copy for the joint
    CK(launch_emit_rows(p->x, p->xln, enc, p->o, p->pmap_dev, nbp, P, E, D, m->bf16, s));
    ++p->launches;
    if (joint) RET(run_joint(p, p->o, nbp * E, E, joint, 1, 0, p->pmap_dev, s));
    CK(launch_advance(p->pos, p->pids_dev, nbp, E, s, p->S, p->status));
    ++p->launches;
    return CAC_OK;
}

// One (sub-)batch step with scratch set `group` on stream s, through the
// graph cache when graphs are enabled (captured on its second sighting).
int step_one(cac_pool* p, int group, int nb, int n, const float* mel, long long mel_bstride, const int* nvalid,
             float* enc, float* joint, int out_bstride, int out_off, const int* ids, cudaStream_t s) {
    use_scratch(p, group);
    if (!p->graphs || p->trace || p->prof) {
        const int r = run_step(p, nb, n, mel, mel_bstride, nvalid, enc, joint, out_bstride, out_off, s, ids);
        use_scratch(p, 0);
        return r;
    }
    GraphKey key{nb, n, nvalid ? 1 : 0, mel, enc, joint, mel_bstride, out_bstride, out_off, ids, group};
    GraphEntry& g = p->gcache[key];
    if (!g.exec) {
        if (g.seen++ == 0) {  // first sighting runs eagerly (sets kernel attributes, warms up)
            const int r = run_step(p, nb, n, mel, mel_bstride, nvalid, enc, joint, out_bstride, out_off, s, ids);
            use_scratch(p, 0);
            return r;
        }
        cudaStream_t cs;
        CK(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
        const long long before = p->launches;
        cudaGraph_t graph = nullptr;
        CK(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal));
        const int r = run_step(p, nb, n, mel, mel_bstride, nvalid, enc, joint, out_bstride, out_off, cs, ids);
        const cudaError_t e = cudaStreamEndCapture(cs, &graph);
        cudaStreamDestroy(cs);
        use_scratch(p, 0);
        const long long captured = p->launches - before;
        p->launches = before;
        if (r != CAC_OK) {
            if (graph) cudaGraphDestroy(graph);
            return r;
        }
        CK(e);
        CK(cudaGraphInstantiate(&g.exec, graph, 0));
        g.kernels = captured;
        cudaGraphDestroy(graph);
    }
    use_scratch(p, 0);
    CK(cudaGraphLaunch(g.exec, s));
    p->launches += g.kernels;
    return CAC_OK;
}

// Concurrent sub-batches of a chunked step over nb streams: flush and traced
// steps and chained steps (the chain kernel keeps its row blocks apart itself)
// run as one batch.  Profiled steps keep the sub-batches, so that per-class
// timings describe the launch configuration of unprofiled steps.
int step_groups(const cac_pool* p, int nb, int n, bool flush) {
    return (p->groups > 1 && !flush && !p->trace && !chain_step_ok(p, nb, n))
               ? std::min(p->groups, (nb + p->group_streams - 1) / p->group_streams)
               : 1;
}

// One chunked step.  Over many streams it runs as up to p->groups concurrent
// sub-batches (contiguous batch slots, <= group_streams each), each on its own
// pool stream with its own scratch and graph, forked from and joined back into
// s; traced, profiled and flush steps stay one batch on s.
int step(cac_pool* p, int nb, int n, const float* mel, long long mel_bstride, const int* nvalid, float* enc,
         float* joint, int out_bstride, int out_off, cudaStream_t s) {
    const int G = step_groups(p, nb, n, nvalid != nullptr);
    if (G <= 1) return step_one(p, 0, nb, n, mel, mel_bstride, nvalid, enc, joint, out_bstride, out_off, p->ids_dev, s);
    const int per = (nb + G - 1) / G;
    const int D = p->m->D, J = p->m->J;
    CK(cudaEventRecord(p->fork_ev, s));
    for (int g = 0; g < G; ++g) {
        const int b0 = g * per, nbg = std::min(per, nb - b0);
        if (nbg <= 0) break;
        CK(cudaStreamWaitEvent(p->gs[g], p->fork_ev, 0));
        if (p->hio_on)  // this sub-batch's mel rows, from the caller's host buffer
            CK(cudaMemcpyAsync(const_cast<float*>(mel) + (size_t)b0 * mel_bstride, p->hio.mel + (size_t)b0 * mel_bstride,
                               (size_t)nbg * mel_bstride * sizeof(float), cudaMemcpyHostToDevice, p->gs[g]));
        RET(step_one(p, g, nbg, n, mel + (size_t)b0 * mel_bstride, mel_bstride, nullptr,
                     enc ? enc + (size_t)b0 * out_bstride * D : nullptr,
                     joint ? joint + (size_t)b0 * out_bstride * J : nullptr, out_bstride, out_off, p->ids_dev + b0,
                     p->gs[g]));
        if (p->hio_on) {  // and its frames back, while the other sub-batches still run
            const size_t eo = (size_t)b0 * out_bstride * D, jo = (size_t)b0 * out_bstride * J;
            if (enc && p->hio.enc)
                CK(cudaMemcpyAsync(p->hio.enc + eo, enc + eo, (size_t)nbg * out_bstride * D * sizeof(float),
                                   cudaMemcpyDeviceToHost, p->gs[g]));
            if (joint && p->hio.joint)
                CK(cudaMemcpyAsync(p->hio.joint + jo, joint + jo, (size_t)nbg * out_bstride * J * sizeof(float),
                                   cudaMemcpyDeviceToHost, p->gs[g]));
        }
        CK(cudaEventRecord(p->join_ev[g], p->gs[g]));
        CK(cudaStreamWaitEvent(s, p->join_ev[g], 0));
    }
    return CAC_OK;
}

}  // namespace

extern "C" int cac_pool_create(cac_model* m, int max_streams, int max_frames_per_step, cac_pool** out) {
    if (!m || !out || max_streams <= 0 || max_frames_per_step <= 0 || max_frames_per_step > 8) return CAC_E_INVAL;
    *out = nullptr;
    cac_pool* p = new (std::nothrow) cac_pool();
    if (!p) return CAC_E_NOMEM;
    auto fail = [&](int code) {
        cac_pool_destroy(p);
        return code;
    };
    p->m = m;
    p->S = max_streams;
    p->nmax = max_frames_per_step;
    const cac_config& c = m->cfg;
    const int pass = c.right_context > 0 ? c.emit_frames + c.lookahead_frames : p->nmax;
    const int rows_per = std::max(pass, p->nmax);
    p->R = ((c.att_left + rows_per + 7) / 8) * 8;
    const int S = p->S, L = m->L, D = m->D, H = m->H, HD = m->HD, F = m->F;
    const size_t ab = act_bytes(m);
    const size_t rows_max = (size_t)S * rows_per;
    const int n = p->nmax;
    p->ring_sstride = (long long)L * H * p->R * HD;
    p->conv_sstride = (long long)L * CONV_CACHE * D;
    p->tail_elems = (size_t)TAIL * MEL;
    int r;
    void* v;
    if ((r = palloc(p, sizeof(int) * S, &v)) != CAC_OK) return fail(r);
    p->pos = static_cast<int*>(v);
    if ((r = palloc(p, sizeof(float) * S * p->tail_elems, &v)) != CAC_OK) return fail(r);
    p->tail = static_cast<float*>(v);
    if ((r = palloc_guarded(p, ab * S * p->ring_sstride, &p->kring)) != CAC_OK) return fail(r);
    if ((r = palloc_guarded(p, ab * S * p->ring_sstride, &p->vring)) != CAC_OK) return fail(r);
    if (m->bf16 && HD == 64 && p->R <= 80) {
        // tensor maps of the tensor-core attention: one copy = one head's ring of
        // one stream and layer (R rows), or one head's position table (NR rows)
        p->amaps.resize(L);
        for (int l = 0; l < L; ++l) {
            AttnMaps& am = p->amaps[l];
            const uint64_t blocks = (uint64_t)S * L * H, bstride = (uint64_t)p->R * HD * 2;
            if (!m->layers[l].has_pmap || !make_tmap_bf16_blocks(&am.k, p->kring, p->R, blocks, bstride, p->R) ||
                !make_tmap_bf16_blocks(&am.v, p->vring, p->R, blocks, bstride, p->R))
                return fail(CAC_E_CUDA);
            am.p = m->layers[l].Pmap;
        }
    }
    if ((r = palloc_guarded(p, ab * S * p->conv_sstride, &p->conv)) != CAC_OK) return fail(r);
    const size_t wsp = m->split ? 2 : 1;  // split windows: rows hi | lo
    // scratch for Ss streams of rows_per rows each
    auto alloc_scratch = [&](int Ss, Scratch& sc) -> int {
        const size_t rows = (size_t)Ss * rows_per;
        void* w;
        int e;
        if ((e = palloc(p, wsp * ab * ((size_t)Ss * (TAIL + 8 * n) + 4) * MEL, &sc.win1)) != CAC_OK) return e;
        if ((e = palloc(p, wsp * ab * ((size_t)Ss * (4 * n + 6) + 4) * D, &sc.win2)) != CAC_OK) return e;
        if ((e = palloc(p, wsp * ab * ((size_t)Ss * (2 * n + 2) + 4) * D, &sc.win3)) != CAC_OK) return e;
        if ((e = palloc(p, wsp * ab * rows * D, &sc.y3)) != CAC_OK) return e;
        if ((e = palloc(p, 4 * rows * D, &w)) != CAC_OK) return e;
        sc.x = static_cast<float*>(w);
        if ((e = palloc(p, ab * rows * D * wsp, &sc.xln)) != CAC_OK) return e;
        if ((e = palloc(p, ab * rows * F * (m->split_ffh ? 2 : 1), &sc.h)) != CAC_OK) return e;
        if ((e = palloc(p, 4 * rows * D, &w)) != CAC_OK) return e;
        sc.q = static_cast<float*>(w);
        if ((e = palloc(p, ab * rows * D * wsp, &sc.o)) != CAC_OK) return e;
        if ((e = palloc(p, ab * rows * D, &sc.glu)) != CAC_OK) return e;
        if ((e = palloc(p, ab * rows * D, &sc.yc)) != CAC_OK) return e;
        if (m->fold_ln) {
            if ((e = palloc(p, sizeof(float2) * rows * (D / 32), &w)) != CAC_OK) return e;
            sc.stats = static_cast<float2*>(w);
        }
        return CAC_OK;
    };
    // concurrent sub-batches of 64 streams for chunked steps (2 .. 4 of them;
    // CAC_GROUPS in the environment sets the count, 1 .. MAX_GROUPS, for tuning)
    const int g_default = std::max(1, std::min(4, S / 64));
    p->groups = c.right_context > 0 ? 1 : std::min(env_int("CAC_GROUPS", g_default, 1, MAX_GROUPS), S);
    p->group_streams = (S + p->groups - 1) / p->groups;
    p->sc.resize(p->groups);
    if ((r = alloc_scratch(S, p->sc[0])) != CAC_OK) return fail(r);
    for (int g = 1; g < p->groups; ++g)
        if ((r = alloc_scratch(p->group_streams, p->sc[g])) != CAC_OK) return fail(r);
    for (int g = 0; g < p->groups && p->groups > 1; ++g) {
        if (cudaStreamCreateWithFlags(&p->gs[g], cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&p->join_ev[g], cudaEventDisableTiming) != cudaSuccess)
            return fail(CAC_E_CUDA);
    }
    if (p->groups > 1 && cudaEventCreateWithFlags(&p->fork_ev, cudaEventDisableTiming) != cudaSuccess)
        return fail(CAC_E_CUDA);
    use_scratch(p, 0);
    if ((r = palloc(p, sizeof(int) * S, &v)) != CAC_OK) return fail(r);
    p->ids_dev = static_cast<int*>(v);
    if ((r = palloc(p, sizeof(int) * S, &v)) != CAC_OK) return fail(r);
    p->rids_dev = static_cast<int*>(v);
    if ((r = palloc(p, sizeof(int) * S, &v)) != CAC_OK) return fail(r);
    p->nvalid_dev = static_cast<int*>(v);
    if ((r = palloc(p, sizeof(int), &v)) != CAC_OK) return fail(r);
    p->status = static_cast<int*>(v);
    if (m->tc) {  // chain counters: completion [phase][row block], exit counter, abort word
        if ((r = palloc(p, sizeof(int) * (CH_MAX_PHASES * CH_MAX_RB + 2), &v)) != CAC_OK) return fail(r);
        p->chain.ctl.cnt = static_cast<int*>(v);
        p->chain.ctl.done = p->chain.ctl.cnt + CH_MAX_PHASES * CH_MAX_RB;
        p->chain.ctl.abort = p->chain.ctl.done + 1;
        p->chain.ctl.status = p->status;
        p->chain.sms = m->sms;
        p->chain.pool = p;
    }
    p->trace_rows = (int)rows_max;
    if (c.right_context > 0) {
        // waiting frames stay below emit + lookahead + one push sub-step
        p->XC = 32;
        if (c.emit_frames + c.lookahead_frames + p->nmax > p->XC || c.emit_frames % 2) return fail(CAC_E_UNSUPPORTED);
        if ((r = palloc(p, sizeof(int) * S, &v)) != CAC_OK) return fail(r);
        p->sub_pos = static_cast<int*>(v);
        if ((r = palloc_guarded(p, sizeof(float) * S * p->XC * D, &v)) != CAC_OK) return fail(r);
        p->x0 = static_cast<float*>(v);
        if ((r = palloc(p, sizeof(int) * S, &v)) != CAC_OK) return fail(r);
        p->pids_dev = static_cast<int*>(v);
        if ((r = palloc(p, sizeof(int) * S, &v)) != CAC_OK) return fail(r);
        p->pmap_dev = static_cast<int*>(v);
    }
    if (cudaHostAlloc(reinterpret_cast<void**>(&p->pinned), sizeof(int) * S * ID_SLOTS, cudaHostAllocDefault) !=
        cudaSuccess)
        return fail(nomem());
    for (int k = 0; k < ID_SLOTS; ++k)
        if (cudaEventCreateWithFlags(&p->slot_ev[k], cudaEventDisableTiming) != cudaSuccess) return fail(CAC_E_CUDA);
    p->alive.assign(S, 0);
    p->finished.assign(S, 0);
    p->pos_host.assign(S, 0);
    p->sub_host.assign(S, 0);
    if (cudaDeviceSynchronize() != cudaSuccess) return fail(CAC_E_CUDA);
    *out = p;
    return CAC_OK;
}

extern "C" void cac_pool_destroy(cac_pool* p) {
    if (!p) return;
    cudaDeviceSynchronize();
    for (auto& kv : p->gcache)
        if (kv.second.exec) cudaGraphExecDestroy(kv.second.exec);
    p->chain.release();
    if (p->chain.ctl.ws) cudaFree(p->chain.ctl.ws);
    if (p->chain.ctl.tcnt) cudaFree(p->chain.ctl.tcnt);
    for (void* d : p->allocs) cudaFree(d);
    if (p->trace_buf) cudaFree(p->trace_buf);
    if (p->pinned) cudaFreeHost(p->pinned);
    if (p->h_mel) cudaFreeHost(p->h_mel);
    if (p->h_out) cudaFreeHost(p->h_out);
    if (p->d_mel) cudaFree(p->d_mel);
    if (p->d_out) cudaFree(p->d_out);
    for (int k = 0; k < ID_SLOTS; ++k)
        if (p->slot_ev[k]) cudaEventDestroy(p->slot_ev[k]);
    for (cudaEvent_t e : p->ev) cudaEventDestroy(e);
    for (int g = 0; g < MAX_GROUPS; ++g) {
        if (p->gs[g]) cudaStreamDestroy(p->gs[g]);
        if (p->join_ev[g]) cudaEventDestroy(p->join_ev[g]);
    }
    if (p->fork_ev) cudaEventDestroy(p->fork_ev);
    delete p;
}

extern "C" int cac_stream_create(cac_pool* p, int* id) {
    if (!p || !id) return CAC_E_INVAL;
    for (int i = 0; i < p->S; ++i) {
        if (!p->alive[i]) {
            // a fresh stream starts at position 0
            CK(cudaDeviceSynchronize());
            const int zero = 0;
            CK(cudaMemcpy(p->pos + i, &zero, sizeof(int), cudaMemcpyHostToDevice));
            if (p->sub_pos) CK(cudaMemcpy(p->sub_pos + i, &zero, sizeof(int), cudaMemcpyHostToDevice));
            p->alive[i] = 1;
            p->finished[i] = 0;
            p->pos_host[i] = 0;
            p->sub_host[i] = 0;
            *id = i;
            return CAC_OK;
        }
    }
    return CAC_E_NOMEM;
}

extern "C" int cac_stream_destroy(cac_pool* p, int id) {
    if (!p || id < 0 || id >= p->S || !p->alive[id]) return CAC_E_INVAL;
    p->alive[id] = 0;
    return CAC_OK;
}

extern "C" int cac_stream_reset(cac_pool* p, int n, const int* ids, void* stream) {
    if (!p) return CAC_E_INVAL;
    if (n == 0) return CAC_OK;
    RET(check_ids(p, n, ids, false));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    RET(upload_ids(p, ids, n, p->rids_dev, s));
    PB(P_RESET);
    CK(launch_set_pos(p->pos, p->rids_dev, n, 0, s, p->S, p->status));
    PE();
    ++p->launches;
    if (p->sub_pos) {
        CK(launch_set_pos(p->sub_pos, p->rids_dev, n, 0, s, p->S, p->status));
        ++p->launches;
    }
    for (int i = 0; i < n; ++i) {
        p->pos_host[ids[i]] = 0;
        p->sub_host[ids[i]] = 0;
        p->finished[ids[i]] = 0;
    }
    return CAC_OK;
}

namespace {

// Subsample `frames` new frames of the listed streams (ids already in
// p->ids_dev) into their x0 rings; mel rows as in run_subsample.  The caller
// keeps frames <= p->nmax, so a ring of XC >= emit + lookahead + nmax rows never
// overwrites a frame that still waits.
int prov_subsample(cac_pool* p, int nb, int frames, const float* mel, long long mel_bstride, const int* nvalid,
                   cudaStream_t s) {
    if (frames > p->nmax) return CAC_E_INVAL;
    RET(run_subsample(p, nb, frames, mel, mel_bstride, nvalid, p->ids_dev, p->sub_pos, s));
    CK(launch_x0_store(p->x, p->x0, p->ids_dev, p->sub_pos, nb, frames, p->XC, p->m->D, s, p->S, p->status));
    CK(launch_advance(p->sub_pos, p->ids_dev, nb, frames, s, p->S, p->status));
    p->launches += 2;
    return CAC_OK;
}

// Run passes for the listed streams.  Rounds of full passes first: every
// stream with emit + lookahead frames waiting takes one (all such streams in
// one batch), until none has.  Final (flush): then each stream's remaining
// frames are drained with truncated lookahead.  Emitted frame i of batch slot b
// lands at row b * out_bstride + n_out[b] + i (n_out[b] grows as it emits).
int prov_drain(cac_pool* p, int n, const int* ids, bool final, float* enc, float* joint, int out_bstride, int* n_out,
               cudaStream_t s) {
    const cac_config& c = p->m->cfg;
    const int E = c.emit_frames, need = c.emit_frames + c.lookahead_frames;
    std::vector<int> pids, prow, slot;
    for (;;) {
        pids.clear();
        prow.clear();
        slot.clear();
        for (int b = 0; b < n; ++b) {
            const int id = ids[b];
            if (p->sub_host[id] - p->pos_host[id] < need) continue;
            if (n_out[b] + E > out_bstride) return CAC_E_INVAL;
            pids.push_back(id);
            prow.push_back(b * out_bstride + n_out[b]);
            slot.push_back(b);
        }
        if (pids.empty()) break;
        RET(upload_ids(p, pids.data(), (int)pids.size(), p->pids_dev, s));
        RET(upload_ids(p, prow.data(), (int)prow.size(), p->pmap_dev, s));
        RET(run_pass(p, (int)pids.size(), need, E, enc, joint, s));
        for (size_t k = 0; k < pids.size(); ++k) {
            p->pos_host[pids[k]] += E;
            n_out[slot[k]] += E;
        }
    }
    if (!final) return CAC_OK;
    for (int b = 0; b < n; ++b) {
        int id = ids[b];
        while (p->sub_host[id] - p->pos_host[id] > 0) {
            const int P = std::min(need, p->sub_host[id] - p->pos_host[id]), Ee = std::min(E, P);
            if (n_out[b] + Ee > out_bstride) return CAC_E_INVAL;
            int row = b * out_bstride + n_out[b];
            RET(upload_ids(p, &id, 1, p->pids_dev, s));
            RET(upload_ids(p, &row, 1, p->pmap_dev, s));
            RET(run_pass(p, 1, P, Ee, enc, joint, s));
            p->pos_host[id] += Ee;
            n_out[b] += Ee;
        }
    }
    return CAC_OK;
}

// Frames subsampled per piece before the passes they enable are run (even, so
// the 160 ms subsampling grid is kept; at most nmax).
int prov_piece(const cac_pool* p) { return std::max(2, (p->nmax / 2) * 2); }

int push_prov(cac_pool* p, int n, const int* ids, const float* mel, int n_mel, float* enc, float* joint, int* n_out,
              cudaStream_t s) {
    const cac_config& c = p->m->cfg;
    if (n_mel <= 0 || n_mel % (8 * c.emit_frames) || n_mel % (8 * c.att_chunk)) return CAC_E_ALIGN;
    const int frames = n_mel / 8;
    RET(upload_ids(p, ids, n, p->ids_dev, s));
    for (int b = 0; b < n; ++b) n_out[b] = 0;
    for (int f0 = 0; f0 < frames;) {
        const int nf = std::min(prov_piece(p), frames - f0);
        RET(prov_subsample(p, n, nf, mel + (size_t)f0 * 8 * MEL, (long long)n_mel * MEL, nullptr, s));
        for (int b = 0; b < n; ++b) p->sub_host[ids[b]] += nf;
        RET(prov_drain(p, n, ids, false, enc, joint, frames, n_out, s));
        f0 += nf;
    }
    return CAC_OK;
}

int flush_prov(cac_pool* p, int n, const int* ids, const float* mel, int mel_stride, const int* n_mel_each,
               float* enc, float* joint, int out_stride, int* n_out_each, cudaStream_t s) {
    const int D = p->m->D, J = p->m->J;
    for (int b = 0; b < n; ++b) {
        const int id = ids[b];
        const int r = n_mel_each[b];
        float* eb = enc ? enc + (size_t)b * out_stride * D : nullptr;
        float* jb = joint ? joint + (size_t)b * out_stride * J : nullptr;
        n_out_each[b] = 0;
        if (r > 0) {
            const float* mb = mel + (size_t)b * mel_stride * MEL;
            RET(upload_ids(p, &id, 1, p->ids_dev, s));
            const int whole = r / 16 * 2;  // frames of whole 160 ms chunks
            for (int f0 = 0; f0 < whole;) {
                const int nf = std::min(prov_piece(p), whole - f0);
                RET(prov_subsample(p, 1, nf, mb + (size_t)f0 * 8 * MEL, (long long)mel_stride * MEL, nullptr, s));
                p->sub_host[id] += nf;
                RET(prov_drain(p, 1, &id, false, eb, jb, out_stride, &n_out_each[b], s));
                f0 += nf;
            }
            const int rem = r - whole * 8;
            if (rem > 0) {
                const int nf = (rem + 7) / 8;
                RET(upload_ids(p, &id, 1, p->ids_dev, s));
                RET(upload_ids(p, &rem, 1, p->nvalid_dev, s));
                RET(prov_subsample(p, 1, nf, mb + (size_t)whole * 8 * MEL, (long long)mel_stride * MEL,
                                   p->nvalid_dev, s));
                p->sub_host[id] += nf;
            }
        }
        RET(prov_drain(p, 1, &id, true, eb, jb, out_stride, &n_out_each[b], s));
        p->finished[id] = 1;
    }
    return CAC_OK;
}

}  // namespace

extern "C" int cac_stream_push(cac_pool* p, int n, const int* ids, const float* mel, int n_mel, float* enc,
                               float* joint, int* n_out, void* stream) {
    if (!p || !mel || !n_out) return CAC_E_INVAL;
    cac_model* m = p->m;
    RET(check_ids(p, n, ids, true));
    if (m->cfg.right_context > 0) return push_prov(p, n, ids, mel, n_mel, enc, joint, n_out, static_cast<cudaStream_t>(stream));
    const int A = m->cfg.att_chunk;
    if (n_mel <= 0 || n_mel % (8 * A)) return CAC_E_ALIGN;
    const int chunk = (p->nmax / A) * A;
    if (chunk <= 0) return CAC_E_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    RET(upload_ids(p, ids, n, p->ids_dev, s));
    const int frames = n_mel / 8;
    for (int f0 = 0; f0 < frames; f0 += chunk) {
        const int nf = std::min(chunk, frames - f0);
        RET(step(p, n, nf, mel + (size_t)f0 * 8 * MEL, (long long)n_mel * MEL, nullptr, enc, joint, frames, f0, s));
    }
    for (int i = 0; i < n; ++i) {
        p->pos_host[ids[i]] += frames;
        n_out[i] = frames;
    }
    return CAC_OK;
}

namespace {
// Host buffers given to a push are page-locked when CUDA knows them as host
// allocations (cudaHostAlloc / cudaHostRegister); those are copied directly.
bool page_locked(const void* ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

// cac_stream_push_host (wait) and cac_stream_push_host_async (!wait).  Both
// queue everything on s; consecutive calls on one pool are ordered on it, so
// the single device staging pair (d_mel, d_out) is never written by one call
// while an earlier call's work still reads it.
int push_host_impl(cac_pool* p, int n, const int* ids, const float* mel, int n_mel, float* enc, float* joint,
                   int* n_out, void* stream, bool wait) {
    if (!p || !mel || !n_out) return CAC_E_INVAL;
    cac_model* m = p->m;
    RET(check_ids(p, n, ids, true));
    if (n_mel <= 0 || n_mel % (8 * m->cfg.att_chunk)) return CAC_E_ALIGN;
    const bool mel_locked = page_locked(mel);
    const bool enc_locked = enc && page_locked(enc), joint_locked = joint && page_locked(joint);
    if (!wait && (!mel_locked || (enc && !enc_locked) || (joint && !joint_locked))) return CAC_E_INVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t mel_n = (size_t)n * n_mel * MEL;
    const int frames = n_mel / 8;
    const size_t enc_n = (size_t)n * frames * m->D, joint_n = (size_t)n * frames * m->J;
    if (mel_n > p->h_mel_cap) {
        CK(cudaStreamSynchronize(s));
        if (p->h_mel) cudaFreeHost(p->h_mel);
        if (p->d_mel) cudaFree(p->d_mel);
        p->h_mel = nullptr;
        p->d_mel = nullptr;
        p->h_mel_cap = 0;
        if (cudaHostAlloc(reinterpret_cast<void**>(&p->h_mel), mel_n * 4, cudaHostAllocDefault) != cudaSuccess ||
            cudaMalloc(&p->d_mel, mel_n * 4) != cudaSuccess)
            return nomem();
        p->h_mel_cap = mel_n;
    }
    if (enc_n + joint_n > p->h_out_cap) {
        CK(cudaStreamSynchronize(s));
        if (p->h_out) cudaFreeHost(p->h_out);
        if (p->d_out) cudaFree(p->d_out);
        p->h_out = nullptr;
        p->d_out = nullptr;
        p->h_out_cap = 0;
        if (cudaHostAlloc(reinterpret_cast<void**>(&p->h_out), (enc_n + joint_n) * 4, cudaHostAllocDefault) !=
                cudaSuccess ||
            cudaMalloc(&p->d_out, (enc_n + joint_n) * 4) != cudaSuccess)
            return nomem();
        p->h_out_cap = enc_n + joint_n;
    }
    // page-locked caller buffers are copied directly, pageable ones staged
    if (!mel_locked) std::memcpy(p->h_mel, mel, mel_n * 4);
    const float* src = mel_locked ? mel : p->h_mel;
    float* he = enc ? (enc_locked ? enc : p->h_out) : nullptr;
    float* hj = joint ? (joint_locked ? joint : p->h_out + enc_n) : nullptr;
    float* de = enc ? p->d_out : nullptr;
    float* dj = joint ? p->d_out + enc_n : nullptr;
    // A synchronous call whose step runs as concurrent sub-batches copies with
    // the sub-batches (each its own slice, on its own stream), so that the
    // frames of the first ones come back while the last still run.  Otherwise,
    // and always in the queued form, one copy in before the push and the
    // frames out after it: measured on 256 streams with pushes queued back to
    // back, the per-sub-batch copies cost 1.451 ms per step against 1.388 for
    // the whole-buffer copies (their latencies sit on every sub-batch's path).
    const int A = m->cfg.att_chunk;
    const bool piped = wait && m->cfg.right_context == 0 && frames <= (p->nmax / A) * A &&
                       step_groups(p, n, frames, false) > 1;
    if (piped) {
        p->hio.mel = src;
        p->hio.enc = he;
        p->hio.joint = hj;
        p->hio_on = true;
        const int r = cac_stream_push(p, n, ids, p->d_mel, n_mel, de, dj, n_out, stream);
        p->hio_on = false;
        RET(r);
    } else {
        CK(cudaMemcpyAsync(p->d_mel, src, mel_n * 4, cudaMemcpyHostToDevice, s));
        RET(cac_stream_push(p, n, ids, p->d_mel, n_mel, de, dj, n_out, stream));
        if (enc) CK(cudaMemcpyAsync(he, de, enc_n * 4, cudaMemcpyDeviceToHost, s));
        if (joint) CK(cudaMemcpyAsync(hj, dj, joint_n * 4, cudaMemcpyDeviceToHost, s));
    }
    if (!wait) return CAC_OK;
    CK(cudaStreamSynchronize(s));
    if (enc && !enc_locked) std::memcpy(enc, p->h_out, enc_n * 4);
    if (joint && !joint_locked) std::memcpy(joint, p->h_out + enc_n, joint_n * 4);
    return CAC_OK;
}
}  // namespace

extern "C" int cac_stream_push_host(cac_pool* p, int n, const int* ids, const float* mel, int n_mel, float* enc,
                                    float* joint, int* n_out, void* stream) {
    return push_host_impl(p, n, ids, mel, n_mel, enc, joint, n_out, stream, true);
}

extern "C" int cac_stream_push_host_async(cac_pool* p, int n, const int* ids, const float* mel, int n_mel,
                                          float* enc, float* joint, int* n_out, void* stream) {
    return push_host_impl(p, n, ids, mel, n_mel, enc, joint, n_out, stream, false);
}

extern "C" int cac_stream_flush_frames(cac_pool* p, int id, int n_mel, int* frames) {
    if (!p || !frames || id < 0 || id >= p->S || n_mel < 0) return CAC_E_INVAL;
    *frames = (n_mel + 7) / 8;
    if (p->m->cfg.right_context > 0) *frames += p->sub_host[id] - p->pos_host[id];  // frames still held back
    return CAC_OK;
}

extern "C" int cac_stream_flush(cac_pool* p, int n, const int* ids, const float* mel, int mel_stride,
                                const int* n_mel_each, float* enc, float* joint, int out_stride, int* n_out_each,
                                void* stream) {
    if (!p || !n_mel_each || !n_out_each) return CAC_E_INVAL;
    cac_model* m = p->m;
    RET(check_ids(p, n, ids, true));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int b = 0; b < n; ++b) {
        const int r = n_mel_each[b];
        int frames = 0;
        RET(cac_stream_flush_frames(p, ids[b], r, &frames));
        if (r < 0 || r > mel_stride || frames > out_stride || (r > 0 && !mel)) return CAC_E_INVAL;
    }
    if (m->cfg.right_context > 0)
        return flush_prov(p, n, ids, mel, mel_stride, n_mel_each, enc, joint, out_stride, n_out_each, s);
    // each stream alone: whole chunks as steps, then the ragged remainder
    const int A = m->cfg.att_chunk;
    const int chunk = (p->nmax / A) * A;
    if (chunk <= 0) return CAC_E_UNSUPPORTED;
    for (int b = 0; b < n; ++b) {
        const int id = ids[b];
        const int r = n_mel_each[b];
        const float* mb = mel ? mel + (size_t)b * mel_stride * MEL : nullptr;
        float* eb = enc ? enc + (size_t)b * out_stride * m->D : nullptr;
        float* jb = joint ? joint + (size_t)b * out_stride * m->J : nullptr;
        RET(upload_ids(p, &id, 1, p->ids_dev, s));
        int done = 0;                        // frames emitted
        const int full = r / (8 * A) * A;    // frames of whole chunks
        while (done < full) {
            const int nf = std::min(chunk, full - done);
            RET(step(p, 1, nf, mb + (size_t)done * 8 * MEL, (long long)mel_stride * MEL, nullptr, eb, jb, out_stride,
                     done, s));
            done += nf;
        }
        const int rem = r - done * 8;
        if (rem > 0) {
            const int nf = (rem + 7) / 8;
            RET(upload_ids(p, &rem, 1, p->nvalid_dev, s));
            RET(step(p, 1, nf, mb + (size_t)done * 8 * MEL, (long long)mel_stride * MEL, p->nvalid_dev, eb, jb,
                     out_stride, done, s));
            done += nf;
        }
        n_out_each[b] = done;
        p->pos_host[id] += done;
        p->finished[id] = 1;
    }
    return CAC_OK;
}

// ===========================================================================
// offline chunked-causal encode
// ===========================================================================
namespace {

// Scratch layout of one offline encode of B windows of up to t_mel_max mel frames.
struct OfflineLayout {
    int T1, T2, T3, W1, W2, W3;
    long long M;
    size_t o_win1, o_win2, o_win3, o_y3, o_x, o_xln, o_h, o_q, o_k, o_v, o_o, o_glu, o_yc, o_mlen, o_flen;
    size_t bytes;
};

OfflineLayout offline_layout(const cac_model* m, int B, int t_mel_max) {
    OfflineLayout y;
    const int D = m->D, F = m->F;
    const size_t ab = act_bytes(m);
    auto half = [](int t) { return (t + 1) / 2; };
    y.T1 = half(t_mel_max);
    y.T2 = half(y.T1);
    y.T3 = half(y.T2);
    y.W1 = 2 + t_mel_max + (t_mel_max & 1);
    y.W2 = 2 + y.T1 + (y.T1 & 1);
    y.W3 = 2 + y.T2 + (y.T2 & 1);
    y.M = (long long)B * y.T3;
    const long long M = y.M;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    };
    const size_t wsp = m->split ? 2 : 1;  // split windows: rows hi | lo
    y.o_win1 = take(wsp * ab * ((size_t)B * y.W1 + 4) * MEL);
    y.o_win2 = take(wsp * ab * ((size_t)B * y.W2 + 4) * D);
    y.o_win3 = take(wsp * ab * ((size_t)B * y.W3 + 4) * D);
    y.o_y3 = take(wsp * ab * M * D);
    y.o_x = take(4 * M * D);
    y.o_xln = take(ab * M * D * (m->split ? 2 : 1));
    y.o_h = take(ab * M * F * (m->split_ffh ? 2 : 1));
    y.o_q = take(4 * M * D);
    y.o_k = take(ab * M * D);
    y.o_v = take(ab * M * D);
    y.o_o = take(ab * M * D * (m->split ? 2 : 1));
    y.o_glu = take(ab * M * D);
    y.o_yc = take(ab * M * D);
    y.o_mlen = take(sizeof(int) * B);
    y.o_flen = take(sizeof(int) * B);
    y.bytes = off;
    return y;
}

int offline_check_args(cac_model* m, int B, const float* mel, const int* mel_len, int t_mel_max, float* enc,
                       int* out_len) {
    if (!m || B <= 0 || !mel || !mel_len || t_mel_max <= 0 || !enc || !out_len) return CAC_E_INVAL;
    for (int b = 0; b < B; ++b)
        if (mel_len[b] < 1 || mel_len[b] > t_mel_max) return CAC_E_INVAL;
    return CAC_OK;
}

// The offline encode on the scratch at `w` (laid out by `lay`); every scratch
// byte that is read is written first in this call, except the zero padding
// rows of the stage-2/3 windows, which are cleared here.
int offline_run(cac_model* m, char* w, const OfflineLayout& lay, int B, const float* mel, const int* mel_len,
                int t_mel_max, float* enc, float* joint, int* out_len, cudaStream_t s) {
    const int D = m->D, F = m->F, L = m->L;
    const size_t ab = act_bytes(m);
    const int bf = m->bf16;
    auto half = [](int t) { return (t + 1) / 2; };
    const int T1 = lay.T1, T2 = lay.T2, T3 = lay.T3, W1 = lay.W1, W2 = lay.W2, W3 = lay.W3;
    const long long M = lay.M;
    const size_t o_win1 = lay.o_win1, o_win2 = lay.o_win2, o_win3 = lay.o_win3, o_y3 = lay.o_y3, o_x = lay.o_x,
                 o_xln = lay.o_xln, o_h = lay.o_h, o_q = lay.o_q, o_k = lay.o_k, o_v = lay.o_v, o_o = lay.o_o,
                 o_glu = lay.o_glu, o_yc = lay.o_yc, o_mlen = lay.o_mlen, o_flen = lay.o_flen;
    void *win1 = w + o_win1, *win2 = w + o_win2, *win3 = w + o_win3, *y3 = w + o_y3, *xln = w + o_xln, *h = w + o_h,
         *kd = w + o_k, *vd = w + o_v, *o = w + o_o, *glu = w + o_glu, *yc = w + o_yc;
    float* x = reinterpret_cast<float*>(w + o_x);
    float* q = reinterpret_cast<float*>(w + o_q);
    int* mlen_d = reinterpret_cast<int*>(w + o_mlen);
    int* flen_d = reinterpret_cast<int*>(w + o_flen);
    long long lc = 0;
    std::vector<int> lens(B);
    for (int b = 0; b < B; ++b) {
        lens[b] = half(half(half(mel_len[b])));
        out_len[b] = lens[b];
    }
    CK(cudaMemcpyAsync(mlen_d, mel_len, sizeof(int) * B, cudaMemcpyHostToDevice, s));
    CK(cudaMemcpyAsync(flen_d, lens.data(), sizeof(int) * B, cudaMemcpyHostToDevice, s));
    CK(cudaStreamSynchronize(s));  // host length arrays must outlive the copies
    const int sp = m->split;
    const int rwm = MEL * (1 + sp), rwd = D * (1 + sp);  // window row widths (split: hi | lo)
    CK(cudaMemsetAsync(win2, 0, ab * ((size_t)B * W2 + 4) * rwd, s));
    CK(cudaMemsetAsync(win3, 0, ab * ((size_t)B * W3 + 4) * rwd, s));
    CK(launch_stage_mel_offline(mel, t_mel_max, mlen_d, win1, W1, B, bf, sp, m->status, s));
    ++lc;
    {
        EpiParams ep;
        ep.kind = EPI_SUB;
        ep.bias = m->sub1.b; ep.out_act = win2; ep.ldo = rwd; ep.split_out = sp ? D : 0;
        ep.P = W1 / 2; ep.T_out = T1; ep.dst_rows = W2; ep.dst_off = 2;
        RET(gemm(m, win1, 2 * rwm, B * (W1 / 2), 3 * MEL, m->sub1, MEL, ep, s, &lc, sp));
        ep.bias = m->sub2.b; ep.out_act = win3;
        ep.P = W2 / 2; ep.T_out = T2; ep.dst_rows = W3; ep.dst_off = 2;
        RET(gemm(m, win2, 2 * rwd, B * (W2 / 2), 3 * D, m->sub2, D, ep, s, &lc, sp));
        ep.bias = m->sub3.b; ep.out_act = y3;
        ep.P = W3 / 2; ep.T_out = T3; ep.dst_rows = T3; ep.dst_off = 0;
        RET(gemm(m, win3, 2 * rwd, B * (W3 / 2), 3 * D, m->sub3, D, ep, s, &lc, sp));
        EpiParams eo;
        eo.kind = EPI_STORE; eo.bias = m->subo.b; eo.out_f32 = x; eo.ldo = D;
        RET(gemm(m, y3, rwd, (int)M, D, m->subo, 0, eo, s, &lc, sp));
    }
    const long long ldl = sp ? 2LL * D : D;  // row stride of the split LayerNorm outputs in xln
    const int shf = m->split_ffh;
    const long long ldh = shf ? 2LL * F : F;  // row stride of the FF hidden activations (split: hi | lo)
    // tensor-core attention: one copy = one head's K (or V) rows of one sequence
    AttnMaps om;
    bool omaps = bf && m->HD == 64 && m->layers[0].has_pmap && m->cfg.right_context == 0;
    if (omaps) {
        const uint32_t box = (uint32_t)attention_offline_box_rows(T3, m->cfg.att_left);
        omaps = box <= 256 && box <= (uint32_t)M && make_tmap_bf16(&om.k, kd, D, M, (uint64_t)D * 2, box) &&
                make_tmap_bf16(&om.v, vd, D, M, (uint64_t)D * 2, box);
    }
    CK(launch_layernorm(x, (int)M, D, m->layers[0].ff1_g, m->layers[0].ff1_b, nullptr, xln, nullptr, nullptr, nullptr,
                        bf, 1 << 30, 0, 0, sp, s));
    ++lc;
    for (int l = 0; l < L; ++l) {
        const LayerW& Lw = m->layers[l];
        EpiParams ep;
        ep.kind = EPI_STORE; ep.act = ACT_SILU; ep.bias = Lw.ff1_w1.b; ep.out_act = h; ep.ldo = ldh; ep.split_out = shf ? F : 0;
        RET(gemm(m, xln, ldl, (int)M, D, Lw.ff1_w1, 0, ep, s, &lc, sp));
        ep = EpiParams(); ep.kind = EPI_RESID; ep.bias = Lw.ff1_w2.b; ep.x = x; ep.ldx = D; ep.scale = 0.5f;
        RET(gemm(m, h, ldh, (int)M, F, Lw.ff1_w2, 0, ep, s, &lc, shf));
        CK(launch_layernorm(x, (int)M, D, Lw.att_g, Lw.att_b, nullptr, xln, nullptr, nullptr, nullptr, bf, 1 << 30, 0,
                            0, sp, s));
        ep = EpiParams(); ep.kind = EPI_QKV; ep.bias = Lw.qkv.b; ep.D = D; ep.HD = m->HD; ep.dense = 1;
        ep.kring = kd; ep.vring = vd; ep.q = q; ep.ldq = D;
        RET(gemm(m, xln, ldl, (int)M, D, Lw.qkv, 0, ep, s, &lc, sp));
        {
            AttnParams a;
            a.q = q; a.ldq = D; a.k = kd; a.v = vd; a.ldk = D;
            a.P = Lw.Ppad; a.rmin = m->rmin; a.NR = m->NR; a.pbu = Lw.pbu; a.pbv = Lw.pbv;
            a.out = o; a.ldo = (int)ldl; a.out_split = sp ? D : 0; a.H = m->H; a.D = D; a.HD = m->HD;
            a.left = m->cfg.att_left; a.chunk = m->cfg.att_chunk; a.rc = m->cfg.right_context;
            a.nb = B; a.T = T3; a.seq_len = flen_d;
            a.scale = 1.f / std::sqrt((float)m->HD);
            AttnMaps lm;
            if (omaps) {
                lm = om;
                lm.p = Lw.Pmap;
                a.maps = &lm;
            }
            CK(launch_attention_offline(a, bf, m->status, s));
        }
        ep = EpiParams(); ep.kind = EPI_RESID; ep.bias = Lw.wo.b; ep.x = x; ep.ldx = D; ep.scale = 1.f;
        RET(gemm(m, o, ldl, (int)M, D, Lw.wo, 0, ep, s, &lc, sp));
        CK(launch_layernorm(x, (int)M, D, Lw.conv_g, Lw.conv_b, nullptr, xln, nullptr, nullptr, nullptr, bf, 1 << 30,
                            0, 0, sp, s));
        ep = EpiParams(); ep.kind = EPI_GLU; ep.bias = Lw.pw1.b; ep.out_act = glu; ep.ldo = D;
        RET(gemm(m, xln, ldl, (int)M, D, Lw.pw1, 0, ep, s, &lc, sp));
        CK(launch_dwconv(glu, nullptr, 0, nullptr, nullptr, T3, 0, Lw.dwT, Lw.bdw, Lw.bng, Lw.bnb, yc, D, B, bf, s));
        ep = EpiParams(); ep.kind = EPI_RESID; ep.bias = Lw.pw2.b; ep.x = x; ep.ldx = D; ep.scale = 1.f;
        RET(gemm(m, yc, D, (int)M, D, Lw.pw2, 0, ep, s, &lc));
        CK(launch_layernorm(x, (int)M, D, Lw.ff2_g, Lw.ff2_b, nullptr, xln, nullptr, nullptr, nullptr, bf, 1 << 30, 0,
                            0, sp, s));
        ep = EpiParams(); ep.kind = EPI_STORE; ep.act = ACT_SILU; ep.bias = Lw.ff2_w1.b; ep.out_act = h; ep.ldo = ldh; ep.split_out = shf ? F : 0;
        RET(gemm(m, xln, ldl, (int)M, D, Lw.ff2_w1, 0, ep, s, &lc, sp));
        ep = EpiParams(); ep.kind = EPI_RESID; ep.bias = Lw.ff2_w2.b; ep.x = x; ep.ldx = D; ep.scale = 0.5f;
        RET(gemm(m, h, ldh, (int)M, F, Lw.ff2_w2, 0, ep, s, &lc, shf));
        if (l + 1 < L)
            CK(launch_layernorm(x, (int)M, D, Lw.out_g, Lw.out_b, x, nullptr, m->layers[l + 1].ff1_g,
                                m->layers[l + 1].ff1_b, xln, bf, 1 << 30, 0, 0, sp, s));
        else
            CK(launch_layernorm(x, (int)M, D, Lw.out_g, Lw.out_b, enc, xln, nullptr, nullptr, nullptr, bf, 1 << 30, 0,
                                0, 0, s));
        lc += 7;
    }
    if (joint) {
        EpiParams ep;
        ep.kind = EPI_STORE; ep.bias = m->joint.b; ep.out_f32 = joint; ep.ldo = m->J;
        RET(gemm(m, xln, D, (int)M, D, m->joint, 0, ep, s, &lc));
    }
    m->launches += lc;
    return CAC_OK;
}

}  // namespace

extern "C" int cac_encode_offline(cac_model* m, int B, const float* mel, const int* mel_len, int t_mel_max, float* enc,
                                  float* joint, int* out_len, void* stream) {
    RET(offline_check_args(m, B, mel, mel_len, t_mel_max, enc, out_len));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const OfflineLayout lay = offline_layout(m, B, t_mel_max);
    if (lay.bytes > m->ws.bytes) {
        CK(cudaStreamSynchronize(s));
        if (m->ws.base) cudaFree(m->ws.base);
        m->ws.base = nullptr;
        m->ws.bytes = 0;
        if (cudaMalloc(&m->ws.base, lay.bytes) != cudaSuccess) return nomem();
        CK(cudaMemset(m->ws.base, 0, lay.bytes));
        m->ws.bytes = lay.bytes;
    }
    return offline_run(m, static_cast<char*>(m->ws.base), lay, B, mel, mel_len, t_mel_max, enc, joint, out_len, s);
}

// ===========================================================================
// offline encode that allocates nothing
// ===========================================================================
namespace {
// Fixed scratch of cac_encode_offline_noalloc: CAC_NOALLOC_SCRATCH_BYTES in
// every device's memory from module load until process exit, shared by all
// calls on that device.  Host code must not use the symbol itself as a device
// address: it is resolved once per device with cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_noalloc_scratch[CAC_NOALLOC_SCRATCH_BYTES];
constexpr int kMaxDevices = 64;
void* g_noalloc_ptr[kMaxDevices] = {};
std::mutex g_noalloc_mu;
}  // namespace

extern "C" int cac_encode_offline_noalloc(cac_model* m, int B, const float* mel, const int* mel_len, int t_mel_max,
                                          float* enc, float* joint, int* out_len, void* stream) {
    RET(offline_check_args(m, B, mel, mel_len, t_mel_max, enc, out_len));
    const OfflineLayout lay = offline_layout(m, B, t_mel_max);
    if (lay.bytes > (size_t)CAC_NOALLOC_SCRATCH_BYTES) return CAC_E_LIMIT;
    int dev = -1;
    CK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return CAC_E_UNSUPPORTED;
    // the array is the current device's: it must be the one holding the weights
    if (dev != m->device) return CAC_E_INVAL;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            // first call on this device (current device): resolve the array's device address
            void* ptr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || !ptr) {
                std::fprintf(stderr, "cac: cudaGetSymbolAddress(scratch) failed: %s\n", cudaGetErrorString(e));
                return CAC_E_CUDA;
            }
            g_noalloc_ptr[dev] = ptr;
        }
        scratch = g_noalloc_ptr[dev];
    }
    return offline_run(m, static_cast<char*>(scratch), lay, B, mel, mel_len, t_mel_max, enc, joint, out_len,
                       static_cast<cudaStream_t>(stream));
}

// ===========================================================================
// state export / import, checks, tracing
// ===========================================================================
namespace {
void act_to_host(const cac_model* m, const void* src_raw, float* dst, size_t n) {
    if (m->bf16) {
        const uint16_t* s = static_cast<const uint16_t*>(src_raw);
        for (size_t i = 0; i < n; ++i) dst[i] = bf2f(s[i]);
    } else {
        std::memcpy(dst, src_raw, n * 4);
    }
}
void host_to_act(const cac_model* m, const float* src, void* dst_raw, size_t n) {
    if (m->bf16) {
        uint16_t* d = static_cast<uint16_t*>(dst_raw);
        for (size_t i = 0; i < n; ++i) d[i] = f2bf(src[i]);
    } else {
        std::memcpy(dst_raw, src, n * 4);
    }
}
}  // namespace

extern "C" int cac_stream_get_state(cac_pool* p, int id, cac_stream_state* st) {
    if (!p || !st || id < 0 || id >= p->S || !p->alive[id]) return CAC_E_INVAL;
    cac_model* m = p->m;
    const int D = m->D, H = m->H, HD = m->HD, L = m->L, R = p->R, left = m->cfg.att_left;
    const size_t ab = act_bytes(m);
    CK(cudaDeviceSynchronize());
    int pos = 0;
    CK(cudaMemcpy(&pos, p->pos + id, sizeof(int), cudaMemcpyDeviceToHost));
    st->subT = pos;
    st->Lc = std::min(pos, left);
    st->finished = p->finished[id];
    st->x0_rows = 0;
    if (p->x0) {
        int sub = 0;
        CK(cudaMemcpy(&sub, p->sub_pos + id, sizeof(int), cudaMemcpyDeviceToHost));
        st->x0_rows = sub - pos;
        if (st->x0)
            for (int i = 0; i < st->x0_rows; ++i)
                CK(cudaMemcpy(st->x0 + (size_t)i * D, p->x0 + ((size_t)id * p->XC + (pos + i) % p->XC) * D,
                              sizeof(float) * D, cudaMemcpyDeviceToHost));
    }
    std::vector<char> raw;
    if (st->mel_tail) {
        if (pos == 0)
            std::fill(st->mel_tail, st->mel_tail + p->tail_elems, 0.f);
        else
            CK(cudaMemcpy(st->mel_tail, p->tail + p->tail_elems * id, sizeof(float) * p->tail_elems,
                          cudaMemcpyDeviceToHost));
    }
    const size_t ring_layer = (size_t)H * R * HD;
    std::vector<float> ring(ring_layer);
    for (int kv = 0; kv < 2; ++kv) {
        float* dst = kv == 0 ? st->k_cache : st->v_cache;
        if (!dst) continue;
        const char* base = static_cast<const char*>(kv == 0 ? p->kring : p->vring) + ab * p->ring_sstride * id;
        raw.resize(ab * ring_layer);
        for (int l = 0; l < L; ++l) {
            CK(cudaMemcpy(raw.data(), base + ab * ring_layer * l, raw.size(), cudaMemcpyDeviceToHost));
            act_to_host(m, raw.data(), ring.data(), ring_layer);
            float* out = dst + (size_t)l * left * D;
            std::fill(out, out + (size_t)left * D, 0.f);
            for (int j = 0; j < st->Lc; ++j) {
                const int pk = pos - st->Lc + j, slot = pk % R;
                for (int hh = 0; hh < H; ++hh)
                    std::memcpy(out + (size_t)j * D + hh * HD, &ring[((size_t)hh * R + slot) * HD], sizeof(float) * HD);
            }
        }
    }
    if (st->conv_cache) {
        const size_t layer = (size_t)CONV_CACHE * D;
        std::vector<float> cc(layer);
        raw.resize(ab * layer);
        const char* base = static_cast<const char*>(p->conv) + ab * p->conv_sstride * id;
        for (int l = 0; l < L; ++l) {
            CK(cudaMemcpy(raw.data(), base + ab * layer * l, raw.size(), cudaMemcpyDeviceToHost));
            act_to_host(m, raw.data(), cc.data(), layer);
            float* out = st->conv_cache + (size_t)l * layer;
            for (int k = 0; k < CONV_CACHE; ++k) {
                const int pk = pos - CONV_CACHE + k;
                if (pk < 0)
                    std::fill(out + (size_t)k * D, out + (size_t)(k + 1) * D, 0.f);
                else
                    std::memcpy(out + (size_t)k * D, &cc[(size_t)(pk & 7) * D], sizeof(float) * D);
            }
        }
    }
    return CAC_OK;
}

extern "C" int cac_stream_set_state(cac_pool* p, int id, const cac_stream_state* st) {
    if (!p || !st || id < 0 || id >= p->S || !p->alive[id] || st->subT < 0) return CAC_E_INVAL;
    cac_model* m = p->m;
    const int D = m->D, H = m->H, HD = m->HD, L = m->L, R = p->R, left = m->cfg.att_left;
    const size_t ab = act_bytes(m);
    const int pos = st->subT, Lc = std::min(pos, left);
    CK(cudaDeviceSynchronize());
    std::vector<char> raw;
    if (st->mel_tail)
        CK(cudaMemcpy(p->tail + p->tail_elems * id, st->mel_tail, sizeof(float) * p->tail_elems,
                      cudaMemcpyHostToDevice));
    const size_t ring_layer = (size_t)H * R * HD;
    std::vector<float> ring(ring_layer, 0.f);
    for (int kv = 0; kv < 2; ++kv) {
        const float* src = kv == 0 ? st->k_cache : st->v_cache;
        if (!src) continue;
        char* base = static_cast<char*>(kv == 0 ? p->kring : p->vring) + ab * p->ring_sstride * id;
        raw.resize(ab * ring_layer);
        for (int l = 0; l < L; ++l) {
            std::fill(ring.begin(), ring.end(), 0.f);
            const float* in = src + (size_t)l * left * D;
            for (int j = 0; j < Lc; ++j) {
                const int pk = pos - Lc + j, slot = pk % R;
                for (int hh = 0; hh < H; ++hh)
                    std::memcpy(&ring[((size_t)hh * R + slot) * HD], in + (size_t)j * D + hh * HD, sizeof(float) * HD);
            }
            host_to_act(m, ring.data(), raw.data(), ring_layer);
            CK(cudaMemcpy(base + ab * ring_layer * l, raw.data(), raw.size(), cudaMemcpyHostToDevice));
        }
    }
    if (st->conv_cache) {
        const size_t layer = (size_t)CONV_CACHE * D;
        std::vector<float> cc(layer, 0.f);
        raw.resize(ab * layer);
        char* base = static_cast<char*>(p->conv) + ab * p->conv_sstride * id;
        for (int l = 0; l < L; ++l) {
            const float* in = st->conv_cache + (size_t)l * layer;
            for (int k = 0; k < CONV_CACHE; ++k) {
                const int pk = pos - CONV_CACHE + k;
                if (pk >= 0) std::memcpy(&cc[(size_t)(pk & 7) * D], in + (size_t)k * D, sizeof(float) * D);
            }
            host_to_act(m, cc.data(), raw.data(), layer);
            CK(cudaMemcpy(base + ab * layer * l, raw.data(), raw.size(), cudaMemcpyHostToDevice));
        }
    }
    CK(cudaMemcpy(p->pos + id, &pos, sizeof(int), cudaMemcpyHostToDevice));
    p->pos_host[id] = pos;
    p->finished[id] = st->finished ? 1 : 0;
    if (p->x0) {
        const int rows = st->x0_rows;
        if (rows < 0 || rows > p->XC || (rows > 0 && !st->x0)) return CAC_E_INVAL;
        for (int i = 0; i < rows; ++i)
            CK(cudaMemcpy(p->x0 + ((size_t)id * p->XC + (pos + i) % p->XC) * D, st->x0 + (size_t)i * D,
                          sizeof(float) * D, cudaMemcpyHostToDevice));
        const int sub = pos + rows;
        CK(cudaMemcpy(p->sub_pos + id, &sub, sizeof(int), cudaMemcpyHostToDevice));
        p->sub_host[id] = sub;
    }
    return CAC_OK;
}

extern "C" int cac_pool_check(cac_pool* p) {
    if (!p) return CAC_E_INVAL;
    CK(cudaDeviceSynchronize());
    int st = 0;
    CK(cudaMemcpy(&st, p->status, sizeof(int), cudaMemcpyDeviceToHost));
    CK(cudaMemset(p->status, 0, sizeof(int)));
    const int st2 = cac_model_check(p->m);
    return st ? st : st2;
}

extern "C" int cac_pool_set_graphs(cac_pool* p, int enable) {
    if (!p) return CAC_E_INVAL;
    p->graphs = enable != 0;
    return CAC_OK;
}

extern "C" long long cac_pool_launch_count(cac_pool* p) { return p ? p->launches : -1; }

extern "C" int cac_pool_check_guards(cac_pool* p) {
    if (!p) return CAC_E_INVAL;
    CK(cudaDeviceSynchronize());
    std::vector<unsigned char> h(GUARD_BYTES);
    for (char* g : p->guards) {
        CK(cudaMemcpy(h.data(), g, GUARD_BYTES, cudaMemcpyDeviceToHost));
        for (unsigned char b : h)
            if (b != 0xFF) return CAC_E_BOUNDS;
    }
    return CAC_OK;
}

extern "C" int cac_build_checked(void) { return kChecked ? 1 : 0; }

extern "C" int cac_pool_sub_batches(cac_pool* p, int n_streams, int n_frames) {
    if (!p || n_streams < 1 || n_streams > p->S || n_frames < 1) return CAC_E_INVAL;
    if (p->m->cfg.right_context > 0) return 1;
    return step_groups(p, n_streams, n_frames, false);
}

extern "C" int cac_pool_set_chains(cac_pool* p, int enable) {
    if (!p) return CAC_E_INVAL;
    if (cudaDeviceSynchronize() != cudaSuccess) return CAC_E_CUDA;
    p->chains = enable != 0;
    return CAC_OK;
}

extern "C" int cac_pool_set_trace(cac_pool* p, int enable) {
    if (!p) return CAC_E_INVAL;
    if (enable && !p->trace_buf) {
        const size_t n = ((size_t)p->m->L * N_TAPS + 1) * p->trace_rows * p->m->D;
        if (cudaMalloc(reinterpret_cast<void**>(&p->trace_buf), n * 4) != cudaSuccess) return nomem();
        CK(cudaMemset(p->trace_buf, 0, n * 4));
    }
    p->trace = enable != 0;
    return CAC_OK;
}

extern "C" int cac_pool_read_trace(cac_pool* p, int layer, int tap, float* host, size_t n_floats) {
    if (!p || !host || !p->trace_buf || tap < 0 || tap > N_TAPS || layer < 0 || layer >= p->m->L) return CAC_E_INVAL;
    const size_t per = (size_t)p->trace_rows * p->m->D;
    if (n_floats > per) return CAC_E_INVAL;
    const float* src = tap == N_TAPS ? p->trace_buf + (size_t)p->m->L * N_TAPS * per
                                     : p->trace_buf + ((size_t)layer * N_TAPS + tap) * per;
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(host, src, n_floats * 4, cudaMemcpyDeviceToHost));
    return CAC_OK;
}

extern "C" int cac_pool_set_profile(cac_pool* p, int enable) {
    if (!p) return CAC_E_INVAL;
    p->prof = enable != 0;
    return CAC_OK;
}

extern "C" int cac_profile_classes(void) { return N_PROF; }

extern "C" const char* cac_profile_class_name(int cls) {
    return (cls >= 0 && cls < N_PROF) ? PROF_NAMES[cls] : nullptr;
}

extern "C" int cac_pool_read_profile(cac_pool* p, int n_classes, double* total_ms, long long* launches) {
    if (!p || !total_ms || !launches || n_classes < N_PROF) return CAC_E_INVAL;
    CK(cudaDeviceSynchronize());
    for (int c = 0; c < n_classes; ++c) {
        total_ms[c] = 0.0;
        launches[c] = 0;
    }
    for (const auto& r : p->rec) {
        float ms = 0.f;
        CK(cudaEventElapsedTime(&ms, p->ev[r.second], p->ev[r.second + 1]));
        total_ms[r.first] += ms;
        launches[r.first] += 1;
    }
    p->rec.clear();
    return CAC_OK;
}

extern "C" int cac_op_gemm_bf16(int M, int N, int K, const void* A, const void* B, const float* bias, float* C,
                                int splits, int a_split, void* stream) {
    if (M < 1 || N < 64 || K < 64 || N % 64 || K % 64 || !A || !B || !C || splits < 0 || splits > 4 ||
        splits > K / 64)
        return CAC_E_INVAL;
    if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C) |
         reinterpret_cast<uintptr_t>(bias)) & 15)
        return CAC_E_ALIGN;
    CUtensorMap ta, tb;
    const uint64_t ka = a_split ? 2ull * K : (uint64_t)K;
    if (!make_tmap_bf16(&ta, A, ka, M, ka * 2, 128) || !make_tmap_bf16(&tb, B, K, N, (uint64_t)K * 2, 64))
        return CAC_E_CUDA;
    EpiParams ep;
    ep.kind = EPI_STORE;
    ep.act_bf16 = 1;
    ep.bias = bias;
    ep.out_f32 = C;
    ep.ldo = N;
    if (splits == 0) splits = choose_splits((N / 64) * ((M + 127) / 128), K / 64);
    CK(launch_gemm_tc(&ta, &tb, M, N, K, 64, 0, splits, a_split ? 1 : 0, ep, nullptr,
                      static_cast<cudaStream_t>(stream)));
    return CAC_OK;
}

extern "C" const char* cac_strerror(int code) {
    switch (code) {
        case CAC_OK: return "ok";
        case CAC_E_INVAL: return "invalid argument";
        case CAC_E_ALIGN: return "push not aligned to the chunk grid (multiple of att_chunk * 8 mel frames)";
        case CAC_E_STATE: return "stream in the wrong state (dead id, or push after flush without reset)";
        case CAC_E_NOMEM: return "out of memory or pool full";
        case CAC_E_CUDA: return "CUDA call failed";
        case CAC_E_DEVICE: return "device-side error";
        case CAC_E_NONFINITE: return "non-finite value in input mel";
        case CAC_E_TIMEOUT: return "bounded device wait gave up";
        case CAC_E_UNSUPPORTED: return "configuration not supported by these kernels";
        case CAC_E_BOUNDS: return "index out of range (checked build) or a pool guard zone overwritten";
        case CAC_E_LIMIT: return "request needs more scratch than the fixed CAC_NOALLOC_SCRATCH_BYTES array";
    }
    return "unknown error";
}
