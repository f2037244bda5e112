// Decode kernel instantiations for 16 token columns (MT = 2), in a
// translation unit of their own so that the library compiles in parallel.
#include "decode_kernel.cuh"

namespace spear {
namespace dec {

DecodeKernelRef kernel_ref_mt2(int NW, int T, bool pc, bool ec) {
  if (NW == 16 && T == 1) return kernel_t<16, 2, 1>(pc, ec);
  return DecodeKernelRef{};
}

}  // namespace dec
}  // namespace spear
