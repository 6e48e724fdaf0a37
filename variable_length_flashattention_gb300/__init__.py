"""GB300-native variable-length FlashAttention forward and paged GQA decode.

The compute path is the CUDA library ``libvfa.so`` (built in-tree for sm_103a)
behind the C ABI declared in ``include/vfa.h``; ``vfa`` is its thin Python
binding.  Importing the package does not load the library: the first call
through ``vfa`` does, and fails loudly if it is missing.
"""
