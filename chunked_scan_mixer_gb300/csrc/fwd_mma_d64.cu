// Instantiations of the tensor-core chunk kernel for d = dv = 64.
#include "fwd_chunk_mma.cuh"

namespace hla2 {

int launch_fwd_chunk_mma_d64(const ChunkArgs& a, int W, int mode, bool cm, cudaStream_t st) {
    switch (W) {
        case 16: return launch_fwd_chunk_mma_t<64, 64, 16>(a, mode, cm, st);
        case 32: return launch_fwd_chunk_mma_t<64, 64, 32>(a, mode, cm, st);
        case 64: return launch_fwd_chunk_mma_t<64, 64, 64>(a, mode, cm, st);
        case 128: return launch_fwd_chunk_mma_t<64, 64, 128>(a, mode, cm, st);
        default: return -2;
    }
}

size_t fwd_chunk_mma_smem_d64(int W, bool cm) {
    switch (W) {
        case 16: return fwd_chunk_mma_smem_t<64, 64, 16>(cm);
        case 32: return fwd_chunk_mma_smem_t<64, 64, 32>(cm);
        case 64: return fwd_chunk_mma_smem_t<64, 64, 64>(cm);
        case 128: return fwd_chunk_mma_smem_t<64, 64, 128>(cm);
        default: return 0;
    }
}

}  // namespace hla2

HLA2_DEBUG_READER(fwd_mma_d64)
