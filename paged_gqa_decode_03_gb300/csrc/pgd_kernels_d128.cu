// Instantiations of the decode kernels for head_dim 128 (block sizes 8 to 128, with and without the page trace, fp16 and quantised pages).
#include "pgd_kernels.cuh"

namespace pgd {

cudaError_t launch_decode_d128(int block_size, bool trace, bool q8, const KVMaps &m,
                              const DecodeParams &p, const LaunchConfig &lc)
{
    return launch_decode_dispatch<128>(block_size, trace, q8, m, p, lc);
}

cudaError_t occupancy_d128(int block_size, int kind, int *ctas_per_sm)
{
    return occupancy_dispatch<128>(block_size, kind, ctas_per_sm);
}

}  // namespace pgd
