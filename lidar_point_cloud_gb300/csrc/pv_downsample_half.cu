// The centroid downsampling kernel built with 512-thread blocks, two resident
// per SM (entry points prepare_downsample_512, downsample_smem_512,
// launch_downsample_512), for clouds whose chunks at one 1024-thread block
// per SM would span several tiles.
#define PV_BLOCK_THREADS 512
#include "pv_downsample.cu"
