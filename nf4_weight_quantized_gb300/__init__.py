"""NF4 weight-quantized projections for GB300 (sm_103a).

``nf4_weight_quantized_gb300.nf4`` is the binding of the C library (loading it
fails loudly when ``libnf4.so`` is not built); ``synth`` holds the seeded input
generators.  This package file imports neither, so the input generators stay
usable on machines without the library.
"""
