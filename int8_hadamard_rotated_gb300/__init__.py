"""GB300-native INT8 convrot linear (sm_103a).

The compute path lives in the CUDA library ``libconvrot.so`` (built from
``csrc/``); ``int8_hadamard_rotated_gb300.ops`` is its thin Python binding.
``workloads`` holds the seeded synthetic inputs. Importing the package does
not load the library; the binding loads it on first use and raises if it is
missing.
"""
__all__ = ["ops", "workloads"]
