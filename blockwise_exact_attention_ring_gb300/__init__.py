"""GB300-native ring-ordered blockwise exact attention.

The compute path is the C-ABI library ``libra.so`` built from ``csrc/``; this
package only marshals arguments to it (see ``binding``).  Importing the package
does not load the library; the first compute call does, and raises if the
library has not been built.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs"]
