"""GB300-native NVFP4 block-scaled GEMM (dense and grouped).

The compute path is the C-ABI library ``libnvfp4gemm.so`` (hand-written sm_103a
CUDA); ``binding`` wraps its entry points with ctypes, argument marshalling
only.  ``workloads`` holds the seeded synthetic problem generators.
"""
