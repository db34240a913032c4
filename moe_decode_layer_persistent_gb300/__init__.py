"""GB300 persistent MoE decode layer: Python binding of the mk_* C ABI.

The compute path is the CUDA library ``libmk.so`` built from ``csrc/``; this
package only marshals arguments (see ``binding``).  Importing a binding call
without the built library raises immediately: there is no CPU fallback.
"""
