// Instantiations of the reverse-mode chunk kernel for d = dv = 16.
#include "bwd_chunk_mma.cuh"

namespace hla2 {

int launch_bwd_chunk_mma_d16(const BwdArgs& a, int W, bool rsum, cudaStream_t st) {
    switch (W) {
        case 16: return launch_bwd_chunk_mma_t<16, 16, 16>(a, rsum, st);
        case 32: return launch_bwd_chunk_mma_t<16, 16, 32>(a, rsum, st);
        case 64: return launch_bwd_chunk_mma_t<16, 16, 64>(a, rsum, st);
        default: return -2;
    }
}

size_t bwd_chunk_mma_smem_d16(int W) {
    switch (W) {
        case 16: return BwdCfg<16, 16, 16>::BYTES;
        case 32: return BwdCfg<16, 16, 32>::BYTES;
        case 64: return BwdCfg<16, 16, 64>::BYTES;
        default: return 0;
    }
}

}  // namespace hla2

HLA2_DEBUG_READER(bwd_mma_d16)
