"""GB300 (sm_103a) W4A8 quantized linear: per-token fp8 activations x MXFP4 / int4-g128 weights,
plus the load-time NVFP4 -> MXFP4 requantizer.  The compute lives in ``libw4a8.so`` (C ABI in
``include/w4a8.h``); ``binding`` is its Python front end and ``synth`` the seeded inputs."""

__all__ = ["binding", "synth", "build"]
