"""Weight-only quantized matrix products (qGEMV / qGEMM) for GB300 (sm_103a).

The compute path is the C-ABI library ``libqmm.so`` (hand-written CUDA); this
package only marshals arguments to it.  See ``qmm.py`` for the Python binding.
"""
