// The variants of the tcgen05 implicit-GEMM kernel for layers with output
// options (a residual, upsample replicas): a translation unit of its own so
// that both halves of the family compile in parallel.
#include "k_igemm_kernel.cuh"

namespace {

template <int BN, int BK, bool SWAP, bool PAIR>
void *fused_ptr(bool flat, bool halo) {
    if (flat) return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, true, SWAP, PAIR, true, false>);
    if (halo) return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, false, SWAP, PAIR, true, true>);
    return reinterpret_cast<void *>(&igemm_bf16_kernel<BN, BK, false, SWAP, PAIR, true, false>);
}

template <int BN, bool SWAP, bool PAIR>
void *fused_bk(int bk, bool flat, bool halo) {
    switch (bk) {
    case 64: return fused_ptr<BN, 64, SWAP, PAIR>(flat, halo);
    case 32: return fused_ptr<BN, 32, SWAP, PAIR>(flat, halo);
    default: return fused_ptr<BN, 16, SWAP, PAIR>(flat, halo);
    }
}

}  // namespace

void *igemm_select_fused(int bn, int bk, bool flat, bool swap, bool pair, bool halo) {
    if (pair) return bn == 128 ? fused_bk<128, false, true>(bk, flat, halo) : fused_bk<256, false, true>(bk, flat, halo);
    if (swap) return fused_bk<128, true, false>(bk, flat, halo);
    switch (bn) {
    case 256: return fused_bk<256, false, false>(bk, flat, halo);
    case 128: return fused_bk<128, false, false>(bk, flat, halo);
    default: return fused_bk<64, false, false>(bk, flat, halo);
    }
}
