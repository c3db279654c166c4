// mk_kernel_hd64.cu — megakernel instances for head dimension 64
// (G = 1..4 query heads per kv head), compiled as their own translation unit.
#include "mk_kernel.cuh"

extern "C" const void *mk_kernel_fn_hd64(int G) {
    switch (G) {
        case 1: return (const void *)mk::mk_megakernel<64, 1>;
        case 2: return (const void *)mk::mk_megakernel<64, 2>;
        case 3: return (const void *)mk::mk_megakernel<64, 3>;
        case 4: return (const void *)mk::mk_megakernel<64, 4>;
        default: return nullptr;
    }
}
