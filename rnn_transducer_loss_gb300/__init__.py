"""rnn_transducer_loss_gb300: fused RNN-T (transducer) loss forward+backward for GB300.

The compute path is a C-ABI shared library (``librnnt_gb300.so``, declared in
``include/rnnt_gb300.h``) of hand-written CUDA kernels for sm_103a.  This
package only marshals arguments to it: ``rnnt_loss`` allocates outputs and the
workspace with PyTorch and passes raw device pointers and the current stream.
The library is loaded on first use and a missing library raises; there is no
other implementation to fall back to.
"""
__all__ = ["rnnt_loss", "RNNTLoss"]


def __getattr__(name):
    if name in ("rnnt_loss", "RNNTLoss"):
        from . import functional
        return getattr(functional, name)
    raise AttributeError(name)
