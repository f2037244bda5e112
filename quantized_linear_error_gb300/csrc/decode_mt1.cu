// Decode kernel instantiations for 8 token columns (MT = 1), in a
// translation unit of their own so that the library compiles in parallel.
#include "decode_kernel.cuh"

namespace spear {
namespace dec {

DecodeKernelRef kernel_ref_mt1(int NW, int T, bool pc, bool ec) {
  if (NW == 16 && T == 1) return kernel_t<16, 1, 1>(pc, ec);
  if (NW == 15 && T == 2) return kernel_t<15, 1, 2>(pc, ec);
  return DecodeKernelRef{};
}

}  // namespace dec
}  // namespace spear
