"""GB300 (sm_103a) PagedAttention decode: a C-ABI CUDA library and its Python binding."""
