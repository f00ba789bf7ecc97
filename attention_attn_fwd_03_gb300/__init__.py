"""GB300-native exact attention: placeholder, replaced by the ctypes binding."""
