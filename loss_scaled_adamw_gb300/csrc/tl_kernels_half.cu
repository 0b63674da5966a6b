// tl_kernels_half.cu - the half-CTA forms of the partial-writing passes: the
// kernels of tl_kernels.cu instantiated with two segments per CTA, and their
// launchers (a second translation unit, so that the two compile side by side).
#define TL_HALF_TU 1
#include "tl_kernels.cu"
