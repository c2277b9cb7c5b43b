// Internal interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace hla2 {

// Arguments of one chunk-kernel launch (summary or output pass of the forward).
struct ChunkArgs {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    int BH, H, n;
    int W;            // chunk width
    int nchunks, seg_chunks, nseg;
    int seg0;         // first segment of this launch (blockIdx.x + seg0)
    int nseg_launch;  // segments in this launch (grid.x)
    const float* gamma;
    int normalize;
    float eps;
    int want_final;
    float* ws;        // forward workspace (floats)
    FwdLayout L;
};

// Tensor-core (mma.sync bf16) chunk kernel: d == dv in {16,32,64,128}, W in {16,32,64,128}.
// Returns 0 on success, -1 on a CUDA error, -2 if the shape is not compiled.
int launch_fwd_chunk_mma(const ChunkArgs& a, int d, int dv, int W, bool summary, bool track_cm,
                         cudaStream_t st);
size_t fwd_chunk_mma_smem(int d, int dv, int W, bool track_cm);  // 0 if not compiled

// SIMT fp32-arithmetic chunk kernel, any d, dv <= 128 (multiples of 8), W <= 128;
// inputs float32 (is_bf16 = false) or bf16.
int launch_fwd_chunk_simt(const ChunkArgs& a, int d, int dv, int W, bool summary, bool track_cm,
                          bool is_bf16, cudaStream_t st);
size_t fwd_chunk_simt_smem(int d, int dv, int W, bool track_cm);

// Inter-segment scan and state conversion kernels (float32).
int launch_init_carry(const ChunkArgs& a, int d, int dv, const float* init_state, cudaStream_t st);
int launch_linear_scan(const float* src, float* dst, int BH, int H, int nsteps, size_t E,
                       size_t src_head_stride, size_t dst_head_stride, bool store_all,
                       const float* gamma, int step_tokens, int power, cudaStream_t st);
int launch_cross(const ChunkArgs& a, int d, int dv, cudaStream_t st);
int launch_finalize(const ChunkArgs& a, int d, int dv, float* final_state, cudaStream_t st);

// Decode step.
int launch_decode_step(float* state, const void* q, const void* k, const void* v, void* out,
                       int N, int H, int d, int dv, const float* gamma, int normalize, float eps,
                       bool is_bf16, cudaStream_t st);

}  // namespace hla2
