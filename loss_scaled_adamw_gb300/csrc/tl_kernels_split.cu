// tl_kernels_split.cu - the split forms of the partial-writing passes: the kernels
// of tl_kernels.cu instantiated with several segments per CTA (kSplitThreads
// threads each), and their launchers (a second translation unit, so that the two
// compile side by side).
#define TL_SPLIT_TU 1
#include "tl_kernels.cu"
