"""GB300-native diffusion-transformer hot path.

The C ABI lives in libdit.so (declared in include/dit.h); its Python binding
is the submodule ``dit`` (importing it fails loudly when the library has not
been built).  ``synth`` draws the seeded synthetic inputs; ``build`` compiles
the library for sm_103a.
"""
