"""GB300-native training-mode Conv -> BatchNorm -> ReLU (CBR) operator.

The compute path is the C-ABI library ``libcbr.so`` built from ``csrc/`` for sm_103a; the
Python binding in :mod:`conv_batchnorm_relu_gb300.cbr` only marshals arguments to it.
Importing this package loads nothing; the library is opened on first use and a missing
library is an error (there is no fallback).
"""
