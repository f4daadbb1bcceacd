"""GB300-native RankMixer block forward: a C-ABI CUDA library (librankmixer.so,
include/rankmixer.h) with a thin Python binding.

    from rankmixer_feature_interaction_gb300.api import RankMixer, token_mix
"""
__all__ = ["api", "synth"]
