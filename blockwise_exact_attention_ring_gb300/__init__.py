"""GB300-native ring-ordered blockwise exact attention.

The compute path is the C-ABI library ``libra.so`` built from ``csrc/`` (see
``include/ra.h``); ``binding`` only marshals arguments to it.  Importing the
package does not load the library; the first compute call does, and raises if
the library has not been built (``build.build()``).
"""
from . import balance, inputs  # noqa: F401
from .binding import (RaError, all_to_all, backward, backward_tile_pairs,  # noqa: F401
                      backward_workspace_bytes, block_units, check, forward, forward_block, forward_ulysses, lib, merge,
                      permute, schedule_stats, schedule_units, set_kernel_variant, status_string,
                      version, workspace_bytes)

__all__ = ["balance", "inputs", "RaError", "all_to_all", "backward", "backward_tile_pairs",
           "backward_workspace_bytes",
           "block_units", "check", "forward",
           "forward_block", "forward_ulysses", "lib", "merge", "permute", "schedule_stats",
           "schedule_units", "set_kernel_variant", "status_string", "version", "workspace_bytes"]
