"""sparse_weight_direct_gb300: direct 2-D convolution with unstructured-sparse
weights on GB300 (sm_103a).  The compute path lives in ``libspconv.so``; this
package is a thin ctypes binding plus host-side accounting helpers."""
