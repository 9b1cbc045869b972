// Launchers of the non-GEMM kernels of the encoder step.
#pragma once

#include "common.cuh"

namespace cac {

// LayerNorm over rows of D (eps 1e-5).  y = LN(x; g1, b1) goes to y_f32
// (row r written at (r / grp) * grp_stride + r % grp + row_off; may alias x
// when the remap is the identity) and/or y_act; when g2 is set, z = LN(y; g2,
// b2) goes to z_act.  act buffers are bf16 when act_bf16, else fp32, with row
// stride D; split (bf16 only) writes them as split operands instead: row
// stride 2D, hi = bf16(v) in columns [0, D), lo = bf16(v - hi) in [D, 2D).
cudaError_t launch_layernorm(const float* x, int M, int D, const float* g1, const float* b1, float* y_f32,
                             void* y_act, const float* g2, const float* b2, void* z_act, int act_bf16, int grp,
                             int grp_stride, int row_off, int split, cudaStream_t s);

// Mel staging: window[b] = [melTail(id) | mel[b]] (14 + 8n rows; tail rows are
// zero when pos[id] == 0), then melTail(id) = last 14 window rows (the tail is
// kept in fp32 [S][14][128]).  mel rows of stream b start at mel + b *
// mel_bstride; rows >= n_valid[b] (if given) read as zero.  Window rows are in
// the activation dtype, 128 wide, or (split, bf16 only) 256 wide: hi | lo.
// Latches CAC_E_NONFINITE on a non-finite mel value.
cudaError_t launch_stage_mel(const float* mel, long long mel_bstride, const int* n_valid, void* win, float* tail,
                             const int* ids, const int* pos, int n, int nb, int act_bf16, int split, int* status,
                             cudaStream_t s, int S = 1 << 30);

// Offline staging: dst[b] = [2 zero rows | mel[b] (rows >= len[b] zero) | pad to W rows],
// rows as in launch_stage_mel.
cudaError_t launch_stage_mel_offline(const float* mel, int t_mel, const int* len, void* dst, int W, int B,
                                     int act_bf16, int split, int* status, cudaStream_t s);

// Tensor maps of the tensor-core streaming attention (see attn_mma.cu): the K
// and V rings as blocks of R rows ((stream * L + layer) * H + head), the
// layer's position table as blocks of NR rows (head).
struct AttnMaps {
    CUtensorMap k, v, p;
};

struct AttnParams {
    const float* q = nullptr;   // fp32 queries, row stride ldq, head h at column h*HD
    int ldq = 0;
    const void* k = nullptr;    // ring base (layer applied) or dense [rows][ldk]
    const void* v = nullptr;
    long long sstride = 0;      // ring: elements between stream ids
    int R = 0;                  // ring rows (streaming)
    int ldk = 0;                // dense row stride (offline)
    const int* ids = nullptr;   // streaming: batch slot -> stream id
    const int* pos = nullptr;   // streaming: stream id -> position of the first query
    int nq = 0;                 // streaming: queries per stream
    const void* P = nullptr;    // position table [H][NR][HD], activation dtype, rel = rmin .. rmin + NR - 1
    int rmin = 0, NR = 0;
    const float* pbu = nullptr; // [H][HD]
    const float* pbv = nullptr;
    void* out = nullptr;        // [rows][ldo], activation dtype
    int ldo = 0;
    int out_split = 0;          // bf16 only, > 0: also write lo = bf16(o - hi) at column out_split + c
    const AttnMaps* maps = nullptr;  // host pointer; tensor-core streaming path only
    int layer = 0, L = 0;            // ring block coordinate (stream * L + layer) * H + head
                                // (a split operand for the out-projection; ldo >= 2 * out_split)
    int H = 0, D = 0, HD = 0;
    int left = 0, chunk = 1, rc = 0;  // rc > 0: window mask [p-left, p+rc]; else chunked mask
    int nb = 0;                 // streaming: batch slots; offline: sequences
    int T = 0;                  // offline: frames per sequence (row stride between sequences)
    const int* seq_len = nullptr;  // offline: valid frames per sequence
    float scale = 1.f;
    int n_streams = 1 << 30;    // streaming (checked build): ids index this many streams
};

// A bounded wait on the K/V copies that gives up latches CAC_E_TIMEOUT in *status.
cudaError_t launch_attention_stream(const AttnParams& a, int act_bf16, int* status, cudaStream_t s);
// Tensor-core variant of the streaming attention (bf16, head_dim 64, <= 4
// queries per stream, <= 80 keys and table rows); launch_attention_stream
// takes it whenever attention_stream_mma_ok holds.
bool attention_stream_mma_ok(const AttnParams& a, int act_bf16);
cudaError_t launch_attention_stream_mma(const AttnParams& a, int* status, cudaStream_t s);
// Tensor-core variant of the offline chunked-causal attention (bf16, head_dim
// 64, chunk <= 4, one block per (head, sequence) with the sequence's K/V
// staged once); maps->k / maps->v: 2-D maps over the dense K / V rows [rows][D]
// with boxes of {64, attention_offline_box_rows(T, left)} rows, maps->p the
// layer's table (as for the streaming path).
bool attention_offline_mma_ok(const AttnParams& a, int act_bf16);
int attention_offline_box_rows(int T, int left);
cudaError_t launch_attention_offline_mma(const AttnParams& a, int* status, cudaStream_t s);
cudaError_t launch_attention_offline(const AttnParams& a, int act_bf16, int* status, cudaStream_t s);

// Causal depthwise conv (k = 9) + affine + SiLU over [conv cache | glu_new].
// Streaming: cache = layer base of [S][L][8][D] rings (stride cs_stride per
// stream id), positions from pos[ids[b]]; the first n_commit GLU rows are
// committed to the cache.  Offline (cache == nullptr): zero left padding,
// nq = frames per sequence, b indexes sequences directly.
cudaError_t launch_dwconv(const void* glu, void* cache, long long cs_stride, const int* ids, const int* pos, int nq,
                          int n_commit, const float* wT, const float* bdw, const float* bng, const float* bnb,
                          void* out, int D, int nb, int act_bf16, cudaStream_t s, int S = 1 << 30,
                          int* status = nullptr);

// Provisional tail: the exact subsampled frames that wait to be emitted live
// in a per-stream ring x0[id][XC][D] (fp32), slot = absolute frame mod XC.
// store:  x0[id][(pos[id] + i) % XC] = x[b * n + i]            (i < n)
// gather: x[b * P + i] = x0[id][(pos[id] + i) % XC]            (i < P)
// emit:   dst[map[b] + i] = x[b * P + i] (map[b] = output row of the first) and
//         act_dst[b * E + i] = act_src[b * P + i]              (i < E)
cudaError_t launch_x0_store(const float* x, float* x0, const int* ids, const int* pos, int nb, int n, int XC, int D,
                            cudaStream_t s, int S = 1 << 30, int* status = nullptr);
cudaError_t launch_x0_gather(const float* x0, float* x, const int* ids, const int* pos, int nb, int P, int XC, int D,
                             cudaStream_t s, int S = 1 << 30, int* status = nullptr);
cudaError_t launch_emit_rows(const float* x, const void* act_src, float* dst, void* act_dst, const int* map, int nb,
                             int P, int E, int D, int act_bf16, cudaStream_t s);

// pos[ids[b]] += n  /  pos[ids[b]] = value
// S, status (checked build): ids index S streams; an id outside latches CAC_E_BOUNDS
cudaError_t launch_advance(int* pos, const int* ids, int nb, int n, cudaStream_t s, int S = 1 << 30,
                           int* status = nullptr);
cudaError_t launch_set_pos(int* pos, const int* ids, int nb, int value, cudaStream_t s, int S = 1 << 30,
                           int* status = nullptr);

// pe[r][2m] = sin(r w_m), pe[r][2m+1] = cos(r w_m), w_m = 10000^(-2m/D), r = rmin + row
cudaError_t launch_sinusoid(float* pe, int NR, int rmin, int D, cudaStream_t s);

// dst fp32 [n] <- src (bf16 or fp32) [n]
cudaError_t launch_to_f32(const void* src, float* dst, long long n, int src_bf16, cudaStream_t s);
// dst[r][c] = hi[r][c] + lo[r][c] of a bf16 split operand [rows][2D]
cudaError_t launch_split_to_f32(const void* src, float* dst, int rows, int D, cudaStream_t s);

}  // namespace cac
