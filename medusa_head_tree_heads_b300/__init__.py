"""B300-native Medusa decode step: heads + top-k, Cartesian candidate tree,
tree-masked attention, verification and acceptance, as a C-ABI CUDA library
(``libmedusa.so``) with a thin ctypes binding."""
