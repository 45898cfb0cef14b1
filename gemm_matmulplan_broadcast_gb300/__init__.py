"""GB300-native ONNX MatMul: a C-ABI CUDA library (``libolc_matmul.so``) and a
thin ctypes binding over it."""
