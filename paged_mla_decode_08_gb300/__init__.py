"""GB300-native paged MLA decode: a C-ABI CUDA library and a thin binding."""
