"""GB300 (sm_103a) fused attention forward: Python side of the C-ABI library.

The compute path is the CUDA library ``libfa_gb300.so`` (kernels under
``csrc/``, declared in ``include/fa.h``).  The binding itself lives in
``attention_forward_blackwell_gb300.binding`` and is loaded lazily so that the
input generators and workload tables can be imported on machines without a
GPU.  There is no CPU fallback: calling the binding without the built library
raises.
"""
