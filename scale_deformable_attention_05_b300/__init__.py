"""B300-native (sm_103a) multi-scale deformable attention (MSDeformAttn).

The operator runs in hand-written CUDA kernels behind the C ABI of
``include/msda.h`` (``libmsda.so``, built by ``build.py``).  ``binding``
marshals torch CUDA tensors into that ABI (plain entry points on sampling
locations and weights; fused ones on reference points, offsets, logits and a
key padding mask); ``module.MSDeformAttn`` is the layer with its projections
around the fused entry points; ``inputs`` draws the seeded synthetic
workloads.  Importing ``binding`` fails loudly when the library has not been
built: there is no CPU fallback.
"""
__version__ = "0.1.0"
