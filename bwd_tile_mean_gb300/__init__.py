"""GB300-native tile-top-k block-sparse video attention (VSA), forward and
backward, behind a C-ABI library (include/vsa.h).

The binding (``bwd_tile_mean_gb300.vsa``) loads the compiled library on
first use; importing this package alone loads nothing.
"""
__all__ = ["inputs", "vsa"]
