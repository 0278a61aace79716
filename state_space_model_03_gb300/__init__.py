"""GB300-native Mamba-1 selective-scan forward, decode step and causal conv1d.

``selective_scan_fn`` (with an optional start state), ``selective_state_update``,
``causal_conv1d_fn`` and ``causal_conv1d_update`` run the hand-written sm_103a
kernels of ``libssfwd.so`` through its C ABI (``include/ssfwd.h``). There is no
CPU fallback: the calls raise if the CUDA library is missing or no GPU is
present.
"""

__all__ = ["selective_scan_fn", "selective_scan_fn_host", "selective_scan_bwd", "SelectiveScanFn",
           "selective_state_update", "causal_conv1d_fn", "causal_conv1d_update"]


def __getattr__(name):
    # Lazy: importing the package (e.g. for the input generator) does not load
    # the CUDA library; the first use of the API does, and fails loudly.
    if name in __all__:
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
