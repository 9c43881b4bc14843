"""GB300-native NVFP4 routed-expert MoE layer: a C-ABI CUDA library
(libmoe_nvfp4.so) and its thin Python binding."""
