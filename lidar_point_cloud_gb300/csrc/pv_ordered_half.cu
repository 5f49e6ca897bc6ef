// The block-tile voxelizer built with 512-thread blocks, two resident per SM
// (entry points prepare_ordered_512, ordered_smem_512, launch_ordered_512).
// Used for clouds whose chunks at one 1024-thread block per SM would span
// several tiles: each SM then runs two blocks, one waiting at a block or
// grid barrier while the other works, and a block's chunk is half as long.
#define PV_BLOCK_THREADS 512
#include "pv_ordered.cu"
