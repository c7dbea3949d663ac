"""SPRINT block-decode step on NVIDIA B300 (sm_103a).

`sprint` binds the C ABI of libsprint.so (include/sprint.h); `decode` holds
the host loop that sequences its calls over a block's denoising steps;
`build` compiles the library.  Importing `sprint` (or using BlockDecoder)
fails if libsprint.so has not been built.
"""
import importlib


def __getattr__(name):
    if name in ("BlockDecoder", "BlockResult"):
        return getattr(importlib.import_module(__name__ + ".decode"), name)
    raise AttributeError(name)
