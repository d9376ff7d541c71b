// launch.h -- internal interface between the C ABI (abi.cu) and the kernel
// translation units.  Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

enum class DType : int { F32 = 0, BF16 = 1, F16 = 2 };

// Warps per CTA of the FP32 record and replay kernels: smaller CTAs, more of
// them per SM, overlap their load, compute and store phases better (measured
// 6 % faster replay and 9 % faster decode record than whole-tile CTAs of
// eight warps).
constexpr int kMaxWarpsPerCta = 4;

// Launch geometry chosen on the host: each CTA owns `rows_cta` consecutive
// value rows (dv) of one (b, hv) state tile; `row_blocks` CTAs cover a tile;
// `tc` timesteps are staged in shared memory at a time.
struct Geometry {
    int threads;        // blockDim.x (a multiple of 32)
    int rows_cta;       // value rows per CTA
    int64_t row_blocks; // ceil(Dv / rows_cta)
    int tc;             // staged chunk length in timesteps
    size_t smem;        // dynamic shared memory bytes
    bool mma;           // record: the tensor-core chunk kernel (bf16 inputs)
};

struct RecordArgs {
    const void *q, *k, *v, *g, *beta;
    const void *state_in;   // f32, or the input type when tstate
    const uint32_t *mask;
    void *y;
    void *state_out;
    void *delta_log, *k_log, *g_log;
    int64_t B, T, Hk, Hv, Dv;
    int rows_cta;
    int64_t row_blocks;
    int tc;
    bool vec_v;     // v rows can be copied in 16-byte pieces (aligned base, Dv*size % 16 == 0)
    bool tiled_gqa; // key head of value head hv: hv % Hk (tiled) instead of hv / (Hv/Hk) (block)
    bool tstate;    // the state is stored in the input type (widened on load, rounded on store)
};

struct ReplayArgs {
    const void *delta_log, *k_log, *g_log;
    const void *state_in;   // f32, or the tape type when tstate
    const uint32_t *mask;
    void *state_out;
    int64_t B, T, Hv, Dv;
    int64_t steps;  // min(accepted, T): steps at or beyond it are never read
    int rows_cta;
    int64_t row_blocks;
    int tc;
    bool vec_d;     // delta_log rows can be copied in 16-byte pieces
    const int32_t *acc_b;  // per-sequence accepted counts [B] (device) or null: then
                           // steps applies to every sequence; else sequence b folds
                           // min(max(acc_b[b], 0), steps) steps
    bool tstate;           // the state is stored in the tape type
};

// Chunked prefill (chunk.cuh): record semantics over chunks of 16 steps,
// with a caller-provided workspace for the chunk-local matrices.
struct ChunkArgs {
    const void *q, *k, *v, *g, *beta;
    const float *state_in;
    const uint32_t *mask;
    void *y;
    float *state_out;
    void *delta_log, *k_log, *g_log;  // delta_log, k_log, g_log may be null
    float *workspace;                 // [B, Hv, nchunks, 544] f32
    int64_t B, T, Hk, Hv, Dv;
    int64_t nchunks;     // ceil(T / 16)
    int64_t row_blocks;  // ceil(Dv / 16)
    bool vec_v;          // v rows can be copied in 16-byte pieces
    bool tiled_gqa;      // key head hv % Hk instead of hv / (Hv/Hk)
};

// Replay as one tensor-core contraction (replay_tc.cuh).
struct ReplayTcArgs {
    const void *delta_log, *k_log, *g_log;
    const float *state_in;
    const uint32_t *mask;
    float *state_out;
    const int32_t *acc_b;  // per-sequence accepted counts or null
    float *w;              // [B, Hv, T] decay weights (workspace)
    float *gam;            // [B, Hv] total decay (workspace)
    float *partial;        // [splits, B, Hv, Dv, Dk] partial sums (workspace) or null
    int64_t B, T, Hv, Dv;
    int64_t steps;         // min(accepted, T) (acc_b null) or T
    int64_t row_blocks;    // ceil(Dv / 128)
    int64_t split_steps;   // steps per split (a multiple of the 16-step stage)
    int splits;            // step splits per tile (1: no partial sums)
    bool staged;           // tape rows are staged with cp.async (16-byte aligned rows)
    unsigned *wait_flag;   // set to 1 when a bounded wait runs out
    long long wait_cycles; // bound on the pipeline's waits
    int inject_expiry;     // testing hook: one wait that nothing completes
};

struct RepeatArgs {
    const void *src;
    void *dst;
    int64_t seq, hg, h, row_bytes;
    int elem_bytes;
    bool vec16;     // rows are whole 16-byte vectors and both bases are 16-byte aligned
};

// Launch geometry for a tile layout with `rows_per_warp` rows per warp (host side).
bool supported_dk(int64_t dk);
int rows_per_warp(int dk);
Geometry record_geometry(int dk, int64_t tiles, int64_t Dv, int64_t T, int esize, bool bf16,
                         int sm_count);
Geometry replay_geometry(int dk, int64_t tiles, int64_t Dv, int64_t steps, int esize,
                         int sm_count);

// One translation unit per element type keeps the (heavily unrolled) kernel
// builds parallel.  Each returns cudaErrorInvalidValue for a Dk it lacks.
cudaError_t launch_record_f32(int dk, const RecordArgs &a, const Geometry &geo, cudaStream_t s);
cudaError_t launch_record_bf16(int dk, const RecordArgs &a, const Geometry &geo, cudaStream_t s);
cudaError_t launch_record_f16(int dk, const RecordArgs &a, const Geometry &geo, cudaStream_t s);
// The tcgen05 record kernel (record_tc.cuh): bf16 calls of at most 16 steps,
// f32 state, Dk = 128, Dv a multiple of 128; its wait-expiry flag (device
// address).
bool record_tc_eligible(const RecordArgs &a, int dk, bool bf16);
cudaError_t launch_record_tc(const RecordArgs &a, int sm_count, cudaStream_t s);
// Read and clear the wait-expiry flag of each tensor-core kernel (host copy,
// synchronous); the bound their pipeline waits use (clock cycles).
cudaError_t record_tc_take_wait_flag(unsigned *was_set);
cudaError_t replay_tc_take_wait_flag(unsigned *was_set);
long long wait_bound_cycles();
int inject_wait_expiry();
cudaError_t launch_replay(DType dt, int dk, const ReplayArgs &a, const Geometry &geo,
                          cudaStream_t s);
// The persistent TMA-fed replay (replay_stream.cuh) for calls of at most 16
// steps with Dk = 128; *launched stays false when the call is not eligible
// (then launch_replay runs), and its wait-expiry flag.
cudaError_t launch_replay_stream(DType dt, int dk, const ReplayArgs &a, int sm_count, cudaStream_t s,
                                 bool *launched);
cudaError_t replay_stream_take_wait_flag(unsigned *was_set);
cudaError_t launch_repeat(const RepeatArgs &a, cudaStream_t s, int sm_count);
cudaError_t launch_chunk(DType dt, int dk, const ChunkArgs &a, cudaStream_t s);
int64_t chunk_workspace_bytes(int64_t B, int64_t T, int64_t Hv);  // -1 on overflow
// The library's static scratch for gdn_chunk_prefill_noalloc (current device).
constexpr size_t kChunkStaticScratchBytes = (size_t)32 << 20;
cudaError_t chunk_static_scratch(float **ptr);
cudaError_t launch_replay_tc(DType dt, int dk, const ReplayTcArgs &a, cudaStream_t s, int sm_count);
// Split plan and workspace bytes of the tensor-core replay (-1 on overflow).
struct ReplayTcPlan {
    int64_t row_blocks, split_steps;
    int splits;
    int64_t w_off, gam_off, partial_off, bytes;
};
ReplayTcPlan replay_tc_plan(int64_t B, int64_t T, int64_t Hv, int64_t Dk, int64_t Dv);

}  // namespace gdn
