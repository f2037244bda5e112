// Decode kernel instantiations for 32 token columns (MT = 4), in a
// translation unit of their own so that the library compiles in parallel.
#include "decode_kernel.cuh"

namespace spear {
namespace dec {

DecodeKernelRef kernel_ref_mt4(int NW, int T, bool pc, bool ec) {
  if (NW == 8 && T == 1) return kernel_t<8, 4, 1>(pc, ec);
  if (NW == 10 && T == 1) return kernel_t<10, 4, 1>(pc, ec);
  if (NW == 12 && T == 1) return kernel_t<12, 4, 1>(pc, ec);
  if (NW == 16 && T == 1) return kernel_t<16, 4, 1>(pc, ec);
  return DecodeKernelRef{};
}

}  // namespace dec
}  // namespace spear
