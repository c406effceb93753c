"""CPU oracle for the layerwise row-band VAE decode -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct float64 restatement of what the decode
computes, written from the ChituDiffusion pages "VAEP：VAE 并行解码" (feature
page) and "Static Layer-Wise VAE Decode" (validation page).  It shares no code
with the CUDA library and never imports it.  Only the test suite, the package
smoke check and the benchmark's CPU-baseline leg may import this package; the
product path never calls it.

Modules
-------
ops      -- the operators one layer at a time (convolution, GroupNorm and its
            per-band central-moment merge, attention, SiLU, RMSNorm, nearest
            upsample, causal temporal conv), each as its plain definition.
decoder  -- the two decoders (AutoencoderKL-style 2D, WanDecoder3d-style
            causal 3D) run either unbanded or literally as the pages' banded
            algorithm (per-layer halo rows, per-band moments merged with the
            weighted rule, band-local Q against gathered K/V).

Pinning: every function here is checked by the CPU tests against something
other than itself -- independent library routines (PyTorch CPU float64
conv2d / conv3d / group_norm / scaled_dot_product_attention / interpolate),
closed forms (delta and shift kernels, constant inputs, law of total
variance), brute force on tiny inputs, and the banded == unbanded invariant.
The one piece with no such pin is the exact Diffusers module wiring of the
two decoders (Diffusers and pretrained weights are not available): the
decoder-level composition is "parity unpinned" against Diffusers, and pinned
only against the written architecture readings.
"""
from . import ops, decoder  # noqa: F401
