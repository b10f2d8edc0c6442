"""Measurement studies that run the library beside a comparison path.

Not part of the library package: the comparison paths here (for example the
eager attention of the peak-memory study) exist only to be measured against.
"""
