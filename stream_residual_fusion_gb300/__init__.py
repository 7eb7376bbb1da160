"""GB300 (sm_103a) single-pass mHC step.

    stream_residual_fusion_gb300.mhc    ctypes binding of libmhc.so (include/mhc.h)
    stream_residual_fusion_gb300.synth  seeded synthetic inputs
    stream_residual_fusion_gb300.build  in-tree build of libmhc.so

Importing the package itself loads nothing; `import stream_residual_fusion_gb300.mhc` loads the
library and fails loudly if it is not built.
"""
