// Kernel instances of the persistent GEMM, one group per compilation of this file
// (GB_INST_GROUP = 0 .. kInstGroups - 1, set by the build), so that the instances compile
// in parallel.  Every launcher the host dispatch (gemm_sm103.cu) calls is instantiated in
// exactly one group.
#include "gemm_launch.cuh"

#ifndef GB_INST_GROUP
#error "GB_INST_GROUP must be defined (0..13)"
#endif

namespace gb {

#define GB_PAIR(BF, IN, SHAPE)                                                               \
  template gb_status prepare_pair<BF, IN, SHAPE>(DeviceState*);                              \
  template gb_status launch_pair<BF, IN, SHAPE>(const Maps&, const Params&, int, cudaStream_t);
#define GB_SINGLE(BF, IN, SHAPE)                                                             \
  template gb_status prepare_single<BF, IN, SHAPE>(DeviceState*);                            \
  template gb_status launch_single<BF, IN, SHAPE>(const Maps&, const Params&, int, cudaStream_t);

#if GB_INST_GROUP == 0      // the 16-bit CTA-pair kernels (the large-problem path)
GB_PAIR(true, kIn16, kShapeStd)
#elif GB_INST_GROUP == 1
GB_PAIR(false, kIn16, kShapeStd)
#elif GB_INST_GROUP == 2    // FP8 inputs, CTA pairs
GB_PAIR(true, kIn8, kShapeStd)
GB_PAIR(false, kIn8, kShapeStd)
#elif GB_INST_GROUP == 3    // block-scaled FP8
GB_PAIR(true, kInMx, kShapeStd)
GB_PAIR(false, kInMx, kShapeStd)
#elif GB_INST_GROUP == 4
GB_SINGLE(true, kInMx, kShapeStd)
GB_SINGLE(false, kInMx, kShapeStd)
#elif GB_INST_GROUP == 5    // single-CTA kernels, 128 x 256 tiles
GB_SINGLE(true, kIn16, kShapeStd)
GB_SINGLE(false, kIn16, kShapeStd)
#elif GB_INST_GROUP == 6
GB_SINGLE(true, kIn8, kShapeStd)
GB_SINGLE(false, kIn8, kShapeStd)
#elif GB_INST_GROUP == 7    // CTA pairs with 256 x 224 tiles
GB_PAIR(true, kIn16, kShapeN224)
GB_PAIR(false, kIn16, kShapeN224)
#elif GB_INST_GROUP == 8
GB_PAIR(true, kIn8, kShapeN224)
GB_PAIR(false, kIn8, kShapeN224)
#elif GB_INST_GROUP == 9    // single-CTA kernels, 128 x 64 tiles (few output columns)
GB_SINGLE(true, kIn16, kShapeNarrow)
GB_SINGLE(false, kIn16, kShapeNarrow)
GB_SINGLE(true, kIn8, kShapeNarrow)
GB_SINGLE(false, kIn8, kShapeNarrow)
#elif GB_INST_GROUP == 10   // CTA pairs with 256 x 512 tiles
GB_PAIR(true, kIn16, kShapeW512)
GB_PAIR(false, kIn16, kShapeW512)
#elif GB_INST_GROUP == 11
GB_PAIR(true, kIn8, kShapeW512)
GB_PAIR(false, kIn8, kShapeW512)
#elif GB_INST_GROUP == 12   // CTA pairs with 256 x 448 tiles
GB_PAIR(true, kIn16, kShapeW448)
GB_PAIR(false, kIn16, kShapeW448)
#elif GB_INST_GROUP == 13
GB_PAIR(true, kIn8, kShapeW448)
GB_PAIR(false, kIn8, kShapeW448)
#else
#error "GB_INST_GROUP out of range"
#endif

}  // namespace gb
