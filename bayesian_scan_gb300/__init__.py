"""GB300 (sm_103a) uncertainty-tracked linear-attention scans.

* ``bayesian_scan_gb300.kdn`` -- the binding of the CUDA library (diagonal
  metaplastic scan with readout, Moebius precision scan);
* ``bayesian_scan_gb300.workloads`` -- seeded synthetic inputs;
* ``bayesian_scan_gb300.build`` -- builds ``_build/libkdn.so`` for sm_103a.

The binding is imported lazily so that the input generators and the build
step work on machines without a GPU.
"""

__all__ = ["kdn", "workloads", "build"]


def __getattr__(name):
    if name in ("kdn", "workloads", "build"):
        import importlib
        return importlib.import_module(f".{name}", __name__)
    raise AttributeError(name)
