"""GB300 (sm_103a) implementation of the Compass-style parallel decoder stack.

The compute lives in libcc.so (C-ABI declared in include/cc.h, built by
``python -m cohere_compass_decoder_gb300.build``); ``_lib`` binds it with ctypes under the
same names and ``model.DecoderStack`` owns device weights and a plan. Importing this
package does not load the library; the first call does, and fails loudly if it was not
built.
"""
from . import _lib  # noqa: F401
from ._lib import CCError, lib  # noqa: F401

__all__ = ["CCError", "lib"]
