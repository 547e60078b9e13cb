// The d <= 128 tensor-core backward with tile-pair accounting (the kernels of
// fa_bwd_tile_pair_count).  They are instantiations of their own, compiled in
// this translation unit (in parallel with the product kernels), so that the
// kernels fa_bwd runs carry no counting code.
#define FA_BWD_SM103_COUNTING 1
#include "fa_bwd_sm103.cu"
