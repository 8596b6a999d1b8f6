// conv_flat.cu -- launches of the flat implicit-GEMM kernel (gemm_flat.cuh)
// planned in conv_gather.cu: the forward of a strided few-channel convolution
// in its space-to-depth form (a stride-1 window whose A operand the tensor
// core reads straight from a TMA box of the channel-blocked copy).  Kept in a
// translation unit of its own so that the library's sources compile in
// parallel.
#include "conv_window.cuh"

namespace cb200 {

template <int BN>
static cudaError_t run_flat(const FlatGeom& fg, const OutGeom& o, const float* img, cudaStream_t st)
{
    ConvFlatProb<BN> p;
    p.terms = math_terms();
    p.fg = fg;
    p.o = o;
    p.bimg = img;
    p.n_tiles = 1;
    p.k_stages = flat_kstages(fg);
    return launch_tc_flat<ConvFlatProb<BN>, BN>(p, fg.Nb * fg.tpi, device_error_word(), st);
}

cudaError_t dispatch_flat(int bn, const FlatGeom& fg, const OutGeom& o, const float* img, cudaStream_t st)
{
    switch (bn) {
    case 16: return run_flat<16>(fg, o, img, st);
    case 32: return run_flat<32>(fg, o, img, st);
    case 48: return run_flat<48>(fg, o, img, st);
    default: return run_flat<64>(fg, o, img, st);
    }
}

}  // namespace cb200
