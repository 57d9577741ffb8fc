"""GB300 (sm_103a) library for absorbed Multi-head Latent Attention decode.

The compute runs in a CUDA shared library with a plain C ABI (``include/mla_decode.h``).
``mla_latent_kv_17_gb300.ops`` is the thin Python binding (argument marshalling only);
it loads the library on first use and raises if the library is missing.
``mla_latent_kv_17_gb300.inputs`` draws the seeded synthetic inputs.
"""
__all__ = ["inputs", "ops"]
