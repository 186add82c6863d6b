"""GB300-native forward pass of one pre-LayerNorm ViT encoder block.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA kernels
(``csrc/``); this package only marshals arguments to it. Importing the package loads
nothing: the library is opened on the first call, and a missing library raises.
"""
__all__ = ["vit_block", "vit_block_ex", "vit_block_host", "load_library"]


def __getattr__(name):
    if name in __all__:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
