"""GB300 (sm_103a) decode step of a W4A8 MXFP4 mixture-of-experts model.

Submodules:

* ``api``      -- the Python binding of the C-ABI library (same entry-point names);
* ``synth``    -- seeded synthetic inputs shaped like the model;
* ``roofline`` -- algorithmic byte / flop counts;
* ``build``    -- compiles ``csrc/`` into the in-tree shared library.

Importing the package loads nothing; ``api`` loads the CUDA library on first use and
raises if it is missing (there is no CPU fallback).
"""
