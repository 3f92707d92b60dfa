"""ReplaySSM decode (Mamba2 and gated delta net) for GB300, behind the C ABI of
librssm.so (include/rssm.h). This package is the thin Python side: the ctypes
binding (same names as the C entry points) and decode-step runners whose buffers
are torch tensors. Every step of the computation runs in the library's CUDA
kernels; importing works without the library, the first call needs it."""
from . import _binding
from ._binding import *  # noqa: F401,F403  (rssm_* entry points, constants, dims structs)
from ._binding import RSSMError, lib  # noqa: F401

__all__ = [n for n in dir(_binding) if n.startswith(("rssm_", "RSSM_"))] + [
    "RSSMError", "Mamba2Dims", "GDNDims", "lib"]


def __getattr__(name):
    # decoder runners import torch; load them lazily
    if name in ("Mamba2ReplayDecoder", "Mamba2FullStateDecoder", "GDNReplayDecoder",
                "GDNFullStateDecoder", "GDNSpecVerifier", "GDNSpecFullStateVerifier",
                "KDAReplayDecoder", "KDAFullStateDecoder", "Mamba2SpecVerifier",
                "torch_dtype_code"):
        from . import decoder
        return getattr(decoder, name)
    raise AttributeError(name)
