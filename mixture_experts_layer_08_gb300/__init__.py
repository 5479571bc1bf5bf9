"""GB300 (sm_103a) Mixture-of-Experts block forward behind a C-ABI CUDA library.

``inputs`` draws seeded synthetic workloads; ``binding`` loads the CUDA library and calls its
C entry points. Importing the package itself loads nothing.
"""
