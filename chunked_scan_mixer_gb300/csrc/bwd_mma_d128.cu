// Instantiations of the reverse-mode chunk kernel for d = dv = 128.
#include "bwd_chunk_mma.cuh"

namespace hla2 {

int launch_bwd_chunk_mma_d128(const BwdArgs& a, int W, bool rsum, cudaStream_t st) {
    switch (W) {
        case 16: return launch_bwd_chunk_mma_t<128, 128, 16>(a, rsum, st);
        case 32: return launch_bwd_chunk_mma_t<128, 128, 32>(a, rsum, st);
        default: return -2;
    }
}

size_t bwd_chunk_mma_smem_d128(int W) {
    switch (W) {
        case 16: return BwdCfg<128, 128, 16>::BYTES;
        case 32: return BwdCfg<128, 128, 32>::BYTES;
        default: return 0;
    }
}

}  // namespace hla2

HLA2_DEBUG_READER(bwd_mma_d128)
