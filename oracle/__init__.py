"""CPU oracle for the FLUX-class AutoencoderKL latent decoder.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run
anything in this package: only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline / reference legs use it. It shares no code with the CUDA
path (no kernels, helpers, constants or layout code) and imports nothing from
it.

Everything is computed in float64 from the definitions in the pages, written
out plainly; see ``vae_oracle`` for the per-function citations.
"""
from .vae_oracle import *  # noqa: F401,F403
