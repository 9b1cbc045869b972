// A chain of projection / LayerNorm phases of the streaming step run by one
// persistent kernel (chain.cu).  Every phase works on the same M rows (the
// step's frames, 128-row blocks); phase p of row block r starts once phase p - 1
// of row block r is complete, so row blocks move through the chain
// independently and no kernel boundary separates the phases.
#pragma once

#include "gemm.cuh"

namespace cac {

enum ChainOp : int { CH_GEMM = 0, CH_LN = 1 };

constexpr int CH_MAX_PHASES = 24;  // phases per chain launch
constexpr int CH_MAX_RB = 64;      // 128-row blocks per chain (M <= 8192)
constexpr int CH_LN_ROWS = 32;     // rows per LayerNorm task

// One phase.  CH_GEMM: C = A B^T with a fused epilogue (gemm.cuh), 128 x 64
// tiles, K split over `splits` tasks whose partials the last one to finish
// adds up.  CH_LN: y = LN(x; g1, b1) to y_f32 (row remap as launch_layernorm)
// and/or y_act, z = LN(y; g2, b2) to z_act (when g2), bf16 act rows, split or
// not.
struct ChainPhase {
    CUtensorMap ta;     // A: bf16 activations [M][K] (or [M][2K] split: hi | lo), 128-row boxes
    CUtensorMap tb;     // B: bf16 weights [N][K], 64-row boxes
    int op = CH_GEMM;
    int K = 0, N = 0, a_split = 0, splits = 1, tiles_n = 0;
    int tasks_rb = 0;   // tasks per row block
    int done_rb = 0;    // completions per row block when the phase is done
    long long ws_off = 0;  // split-K partials: first float in the workspace
    int tc_off = 0;        // split-K tile counters: first counter
    EpiParams ep;
    // CH_LN
    const float* x = nullptr;
    const float *g1 = nullptr, *b1 = nullptr, *g2 = nullptr, *b2 = nullptr;
    float* y_f32 = nullptr;
    bf16* y_act = nullptr;
    bf16* z_act = nullptr;
    int D = 0, grp = 1 << 30, grp_stride = 0, row_off = 0, split = 0;
};

// Device state of a chain launch: per (phase, row block) completion counters,
// split-K tile counters, the workspace of the split-K partials, an exit counter
// and an abort word.  The last CTA to leave zeroes the completion counters, so
// consecutive launches (stream-ordered) start from zero.
struct ChainCtl {
    int* cnt = nullptr;     // [CH_MAX_PHASES][CH_MAX_RB]
    int* tcnt = nullptr;    // split-K tile counters
    int* done = nullptr;    // [1]
    int* abort = nullptr;   // [1]
    float* ws = nullptr;
    int* status = nullptr;
};

// Split-K partial floats a phase needs (0 when splits == 1).
inline long long chain_ws_floats(const ChainPhase& p, int n_rb) {
    return p.op == CH_GEMM && p.splits > 1 ? (long long)n_rb * p.tiles_n * p.splits * 128 * 64 : 0;
}

// One cooperative launch of `grid` CTAs (one per SM) over the n_phases phases
// at d_phases (device memory) for M rows.
cudaError_t launch_chain(const ChainPhase* d_phases, int n_phases, int M, const ChainCtl& ctl, int grid,
                         cudaStream_t s);

// Dynamic shared memory of the chain kernel (bytes).
int chain_smem_bytes();

}  // namespace cac
