"""GB300-native CTR sparse-embedding + dot-interaction path.

The compute lives in the CUDA library ``libctr.so`` (C-ABI, declared in
``include/ctr.h``); ``sparse_embeddings_feature_gb300.ctr`` is its thin Python
binding.  ``workload`` draws the seeded synthetic inputs.  Importing this
package loads nothing; the library is loaded on first use of ``ctr``.
"""
