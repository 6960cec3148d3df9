// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units. Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace rn {

enum DType { kF32 = 0, kF16 = 1, kBF16 = 2 };

inline int elem_bytes(int dt) { return dt == kF32 ? 4 : 2; }

// One backward problem, already validated by the API layer.
struct BwdProblem {
    const void *x;        // x (plain) or added (fused-add)
    const void *gamma;
    const void *dy;
    const float *rstd;
    const void *dres;     // nullable
    void *dx;
    float *dw_f32;
    void *dw_cast;        // nullable
    uint8_t *ws;          // workspace (header + partial rows)
    int64_t M;
    int N;
    int dtype;
};

// Launch shape of the row engine.
struct RowPlan {
    int cpt;           // 16-byte chunks per thread per row (1, 2, 4)
    int team_threads;  // threads that share one row (multiple of 32)
    int teams;         // rows processed concurrently per CTA
    int stages;        // async-copy ring depth per thread (rows in flight + 1)
    int grid;          // CTAs (persistent)
    size_t smem;       // dynamic shared memory bytes
    bool atomic;       // weight gradient via fp32 atomics (else scratch partials)
};

// Launch shape of the cluster engine (rows longer than one CTA's tile).
struct ClusterPlan {
    int csize;         // CTAs per cluster (2..16)
    int slice;         // 16-byte chunks of a row per CTA
    int cpt;           // chunks per thread (1, 2, 4)
    int threads;       // threads per CTA (multiple of 32, <= 512)
    int stages;        // async-copy ring depth per thread
    int clusters;      // clusters launched (persistent)
    size_t smem;       // dynamic shared memory bytes per CTA
    bool atomic;
};

struct GenericPlan {
    int threads;       // CTA size
    int grid;
    bool smem_dw;      // per-CTA weight-gradient partial in shared memory
    size_t smem;
    bool atomic;
    int rows = 0;      // vector variant: rows in flight per CTA iteration (2, 4); 0 = scalar
    int cpb = 0;       // realigning engine: column blocks per thread (2, 4); 0 = not used
    int phase = 0;     // phase-class kernel: 16-byte chunks per thread (1, 2); 0 = not used
    int phase_rows = 1;  // phase-class kernel: rows per CTA iteration (1, 2)
    bool prefetch = false;  // phase-class kernel: L2 prefetch two iterations ahead
};

// Launch shape of the staged phase-class kernel (rows that are not 16-byte
// multiples, staged in shared memory by bulk copies).
struct StagePlan {
    int cpt;           // 16-byte chunks per thread (1, 2, 4)
    int team_threads;  // threads that share one row (multiple of 32)
    int teams;         // rows in progress per CTA (1..15)
    int slots;         // shared-memory slots per team (2..4): rows in flight + 1
    int grid;          // CTAs (persistent)
    size_t smem;       // dynamic shared memory bytes
    bool atomic;
    int64_t skip_row = -1;  // test hook (see RN_OPT_TEST_WAIT_TIMEOUT); -1 = off
};

// Row engine: largest chunk count per row and CTA thread cap for a cpt.
constexpr int kRowMaxChunks = 2048;
int row_max_threads(int cpt);
size_t row_smem_bytes(int teams, int stages, int ntensors, int team_chunks);
size_t generic_smem_bytes(int N, bool smem_dw);
size_t generic_vec_smem_bytes(int N);

cudaError_t launch_bwd_row(const BwdProblem &p, const RowPlan &plan, cudaStream_t s,
                           bool pdl_after_zero);
cudaError_t launch_bwd_generic(const BwdProblem &p, const GenericPlan &plan, cudaStream_t s,
                               bool pdl_after_zero);
// Rows that are not 16-byte multiples, all row tensors at one alignment phase.
int phase_period(int N, int dtype);
int phase_blocks_per_sm(int dtype, bool dres, bool atomic, int cpt, int rows, int threads);
size_t ln_phase_smem_bytes(int N, bool atomic);
int ln_phase_blocks_per_sm(int dtype, bool atomic, int cpt, int threads, size_t smem);
cudaError_t launch_bwd_phase(const BwdProblem &p, const GenericPlan &plan, cudaStream_t s,
                             bool pdl_after_zero);
// Staged phase-class kernel: its shared memory for a tile (the ring, or the
// teams' weight-gradient regions if larger), and the per-tensor slot size and
// one team's region in words it lays out.
uint32_t stage_ring_offset(int slots);
size_t stage_smem_bytes(int N, int dtype, bool dres, int teams, int slots, int cpt,
                        int team_threads, uint32_t *tensor_bytes, uint32_t *region_words);
// Resident CTAs per SM of one instance at a CTA size and dynamic shared memory.
int stage_blocks_per_sm(int dtype, bool dres, bool atomic, int cpt, int threads, size_t smem);
cudaError_t launch_bwd_stage(const BwdProblem &p, const StagePlan &plan, cudaStream_t s,
                             bool pdl_after_zero);
// Read and clear the device status word (bit 0: a bounded wait in a kernel ran
// out); synchronizes the device first. The LayerNorm and forward staged
// kernels keep their own words (device variables are per translation unit),
// read and cleared by the other two calls without synchronizing.
cudaError_t take_device_status(unsigned int *status);
cudaError_t take_ln_device_status(unsigned int *status);
cudaError_t take_fwd_device_status(unsigned int *status);
size_t realign_smem_bytes(int N, int dtype, int rows, bool dres);
cudaError_t launch_bwd_realign(const BwdProblem &p, const GenericPlan &plan, cudaStream_t s,
                               bool pdl_after_zero);
size_t cluster_smem_bytes(int stages, int ntensors, int cpt, int threads);
// Clusters of plan's shape that fit on the device at once (occupancy query).
cudaError_t cluster_max_active(const BwdProblem &p, const ClusterPlan &plan, int *clusters);
cudaError_t launch_bwd_cluster(const BwdProblem &p, const ClusterPlan &plan, cudaStream_t s,
                               bool pdl_after_zero);
// Scratch mode: dw_f32 = sum of G partial rows (fixed order), optional cast;
// either output may be NULL.
cudaError_t launch_finalize(const float *partials, int G, int N, float *dw_f32, void *dw_cast,
                            int dtype, cudaStream_t s, bool pdl);
// The same over partial rows of ld floats holding two length-N outputs side
// by side (dw2_f32 and dw2_cast both NULL: one output).
cudaError_t launch_finalize2(const float *partials, int G, int ld, int N, float *dw_f32,
                             void *dw_cast, float *dw2_f32, void *dw2_cast, int dtype,
                             cudaStream_t s, bool pdl);
// Atomic mode: zero before the row pass, cast after it (second buffers nullable).
cudaError_t launch_zero_f32(float *p, int N, cudaStream_t s, float *p2 = nullptr);
cudaError_t launch_cast(const float *dw_f32, void *dw_cast, int N, int dtype, cudaStream_t s,
                        bool pdl, const float *dw2_f32 = nullptr, void *dw2_cast = nullptr);

struct FwdProblem {
    const void *x;
    const void *residual;  // nullable: plain forward
    const void *gamma;
    void *y;
    void *residual_out;    // fused-add only
    float *rstd;           // nullable
    float eps;
    int64_t M;
    int N;
    int dtype;
};

// Unaligned rows (and rows longer than the row engine's tile): one CTA per row.
cudaError_t launch_fwd(const FwdProblem &p, int num_sms, cudaStream_t s);

// Forward row engine (aligned rows): RMSNorm, fused-add RMSNorm, LayerNorm.
enum FwdMode { kFwdRms = 0, kFwdFused = 1, kFwdLn = 2 };
struct FwdRowProblem {
    int mode;
    const void *x;
    const void *residual;   // fused-add
    const void *gamma;
    const void *beta;       // LayerNorm, nullable
    void *y;
    void *residual_out;     // fused-add
    float *mean;            // LayerNorm, nullable
    float *rstd;            // nullable
    float eps;
    int64_t M;
    int N;
    int dtype;
};
size_t fwd_row_smem_bytes(int teams, int stages, int ntensors, int team_chunks);
cudaError_t launch_fwd_row(const FwdRowProblem &p, const RowPlan &plan, cudaStream_t s);
// Aligned rows longer than the row engine's tile: one CTA per row, 16-byte loads.
cudaError_t launch_fwd_long(const FwdRowProblem &p, int num_sms, cudaStream_t s);
// Rows that are not 16-byte multiples, row tensors at one alignment phase and
// gamma (beta) 16-byte aligned: 16-byte chunks plus element-wise head and tail.
bool fwd_generic_vec_ok(const FwdRowProblem &p);
// The same rows, each CTA on one alignment class of rows (row tensors at one
// phase, at most 1024 whole 16-byte chunks; gamma and beta at any alignment).
bool fwd_phase_ok(const FwdRowProblem &p);
cudaError_t launch_fwd_phase(const FwdRowProblem &p, int cpt, int grid, int threads,
                             cudaStream_t s);
cudaError_t launch_fwd_generic_vec(const FwdRowProblem &p, int num_sms, cudaStream_t s);
// The same rows staged in shared memory by per-warp bulk copies (row tensors
// at one phase, at most 2048 whole 16-byte chunks; gamma and beta at any
// alignment): the backward staged kernel's work split, with the forward math.
bool fwd_stage_ok(const FwdRowProblem &p);
size_t fwd_stage_smem_bytes(int N, int dtype, int mode, int teams, int slots);
int fwd_stage_blocks_per_sm(int dtype, int mode, int cpt, int threads, size_t smem);
cudaError_t launch_fwd_stage(const FwdRowProblem &p, const StagePlan &plan, cudaStream_t s);

// LayerNorm.
struct LnFwdProblem {
    const void *x;
    const void *gamma;
    const void *beta;      // nullable: no bias
    void *y;
    float *mean;           // nullable
    float *rstd;           // nullable
    float eps;
    int64_t M;
    int N;
    int dtype;
};

struct LnBwdProblem {
    const void *x;
    const void *gamma;
    const void *dy;
    const float *mean;
    const float *rstd;
    void *dx;
    float *dg_f32;
    float *db_f32;         // nullable: no bias gradient
    void *dg_cast;         // nullable
    void *db_cast;         // nullable
    uint8_t *ws;           // workspace (header + partial rows of 2N floats)
    int64_t M;
    int N;
    int dtype;
};

cudaError_t launch_ln_bwd_phase(const LnBwdProblem &p, const GenericPlan &plan, cudaStream_t s,
                                bool pdl_after_zero);
// LayerNorm staged phase-class kernel (at most 1024 whole chunks a row, 1 or 2
// chunks a thread): shared memory of a tile and the launch.
uint32_t ln_stage_ring_offset(int slots);
size_t ln_stage_smem_bytes(int N, int dtype, int teams, int slots, uint32_t *tensor_bytes,
                           uint32_t *region_words);
int ln_stage_blocks_per_sm(int dtype, bool atomic, int cpt, int threads, size_t smem);
cudaError_t launch_ln_bwd_stage(const LnBwdProblem &p, const StagePlan &plan, cudaStream_t s,
                                bool pdl_after_zero);

// LayerNorm forward for unaligned rows (and rows longer than the row engine's tile).
cudaError_t launch_ln_fwd(const LnFwdProblem &p, int num_sms, cudaStream_t s);
// Default chunks-per-thread cap of the LayerNorm row engine (two fp32
// accumulators per element pair instead of one).
constexpr int kLnMaxCpt = 2;
int ln_row_max_threads(int cpt);
size_t ln_row_smem_bytes(int teams, int stages, int team_chunks);
size_t ln_generic_smem_bytes(int N, bool smem_dw);
size_t ln_generic_vec_smem_bytes(int N);
cudaError_t launch_ln_bwd_row(const LnBwdProblem &p, const RowPlan &plan, cudaStream_t s,
                              bool pdl_after_zero);
cudaError_t launch_ln_bwd_generic(const LnBwdProblem &p, const GenericPlan &plan,
                                  cudaStream_t s, bool pdl_after_zero);
size_t ln_cluster_smem_bytes(int stages, int cpt, int threads);
cudaError_t ln_cluster_max_active(const LnBwdProblem &p, const ClusterPlan &plan, int *clusters);
cudaError_t launch_ln_bwd_cluster(const LnBwdProblem &p, const ClusterPlan &plan, cudaStream_t s,
                                  bool pdl_after_zero);

// Replace the calling thread's message returned by rn_last_error().
void set_last_error(const char *msg);

// Set the dynamic shared memory cap of a kernel once per device.
cudaError_t ensure_smem_attr(const void *func, size_t bytes);

}  // namespace rn
